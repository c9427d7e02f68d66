"""The multi-process path of the benchmark on CPU (gloo, world size 2): each
rank scores a token-balanced, contiguous share of one corpus, the per-rank
scores concatenate to the single-process result, and the step time is the
maximum over ranks. The CPU oracle stands in for the GPU kernel here; the
sharding and the reductions are what is tested."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_shard_documents_partition_and_balance():
    rng = np.random.default_rng(0)
    for world in (1, 2, 3, 8):
        lens = rng.integers(0, 300, size=1000)
        lens[::17] = 0  # empty documents anywhere
        ranges = [bench.shard_documents(lens, r, world) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == len(lens)
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a1 == b0 and a0 <= a1
        tokens = [int(lens[a:b].sum()) for a, b in ranges]
        assert max(tokens) - min(tokens) <= 2 * lens.max()  # whole documents: within two documents of even


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from datagen import workloads
        w = workloads.make("colbert_varlen", Nq=2, Lq=8, Nd=40, ld_min=0, ld_max=30, dim=16)
        j0, j1 = bench.shard_documents(w["lens"], rank, world)
        cu = w["cu_seqlens_d"].astype(np.int64)
        q_off = np.arange(w["Nq"] + 1, dtype=np.int64) * w["Lq"]
        docs = np.arange(j0, j1, dtype=np.int64)
        s, _, _ = oracle.fwd_packed(w["Q"].reshape(-1, 16), q_off, w["D"], cu, "f16", docs=docs, threads=1)
        parts = [None] * world
        dist.all_gather_object(parts, (j0, j1, s))
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        units = torch.tensor([float(j1 - j0)], dtype=torch.float64)
        dist.all_reduce(units, op=dist.ReduceOp.SUM)
        if rank == 0:
            full, _, _ = oracle.fwd_packed(w["Q"].reshape(-1, 16), q_off, w["D"], cu, "f16", threads=1)
            parts.sort(key=lambda p: p[0])
            assert parts[0][0] == 0 and parts[-1][1] == w["Nd"]
            joined = np.concatenate([p[2] for p in parts], axis=1)
            assert np.array_equal(joined, full)
            assert float(t[0]) == float(world)          # maximum over ranks
            assert float(units[0]) == float(w["Nd"])     # documents summed over ranks
            open(os.path.join(out_dir, "ok"), "w").write("ok")
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_gloo_sharded_scores(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    assert (tmp_path / "ok").exists()
