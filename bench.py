#!/usr/bin/env python3
"""MaxSim throughput on one GB300 (docs scored / s) with its roofline.

Default workload (the one the headline line reports): ColBERT rerank over
packed documents -- Nq = 32 queries of Lq = 32 tokens, Nd = 100,000 documents
with lengths uniform in [32, 300], dim = 128, f16, l2-normalised Gaussian rows
(seeded, synthetic). A step is one maxsim_fwd_varlen call scoring every
document against every query.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--shard weak|global]

Other workloads (measured the same way, for the design notes):
  chamfer_100k     Chamfer distance, forward + backward, of two 100,000-point
                   3-D clouds (float32): cloud pairs/s, fp32 ALU roofline
  tiny_rerank      1 x 32 tokens vs 1,000 x 180 (f16), scores + argmax
  colpali_cross    128 x 128 vs 128 x 1024 (bf16), masks, scores + argmax
  contrastive_bwd  the backward of 64 x 128 vs 64 x 1024 (bf16)
  int8_rerank      1 x 1024 vs 10,000 x 1024 (INT8, per-token scales)
  two_stage_topk   32 x 32 vs 100,000 x 128: INT8 scores, top 1,000, f16
                   rescoring, top 100 (docs/s)
  colpali_out_of_core  1 x 32 vs 100,000 x 1024 (bf16, 26 GB) streamed from
                   page-locked host memory in 20,000-document blocks
Inputs smaller than L2 are timed step by step with an L2 flush between steps.

Prints one JSON line (rank 0). Under torchrun every rank scores its own
documents (--shard weak, the default: per-GPU work fixed) or its token-balanced
share of one corpus (--shard global); there is no communication on the data
path, and the time is the maximum over ranks between barriers.

--impl reference times the CPU oracle (test infrastructure) on bounded samples
of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MaxSim docs scored/s at 1 GB300 + % of roofline (HBM GB/s or tensor-pipe)"
UNIT = "docs/s"
CHAMFER_METRIC = "Chamfer distance forward + backward of 100K-point cloud pairs/s at 1 GB300 + % of roofline"
CHAMFER_UNIT = "cloud pairs/s"
FP32_LANES_PER_SM = 128  # fp32 FMA lanes per SM (4 sub-partitions x 32)


def metric_of(workload: str):
    return (CHAMFER_METRIC, CHAMFER_UNIT) if workload.startswith("chamfer") else (METRIC, UNIT)


def chamfer_fma(B: int, N: int, M: int, dim: int) -> int:
    """FMAs of the nearest-point search: dim per (source, target) pair, both
    directions (the min of each pair is extra)."""
    return 2 * B * N * M * dim
L2_BYTES = 129 * 1024 * 1024
NOMINAL_BF16_TFLOPS = 2250.0     # GB300 dense bf16 / f16 (vendor figure, context beside the measured peak)
NOMINAL_HBM_GBS = 7900.0         # GB300 HBM3e (vendor figure)
TENSOR_FLOP_PER_CYCLE_SM = 8192  # f16 MMA M=128 N=128 K=16 in 64 cycles

# ---------------------------------------------------------------- byte / flop accounting

def io_naive_bytes(nq_tok: int, nd_tok: int, d: int, B: int, elem: int = 2, s_bytes: int = 4) -> int:
    """HBM bytes of the materialise-then-reduce path for one query against B
    documents: read Q, read D, write and read back S ("TileMaxSim" Sec. 2.3,
    Eq. (4))."""
    return nq_tok * d * elem + B * nd_tok * d * elem + 2 * B * nq_tok * nd_tok * s_bytes


def io_fused_bytes(nq_tok: int, nd_tok: int, d: int, B: int, elem: int = 2, out_bytes: int = 4) -> int:
    """HBM bytes of the fused path as that page counts them: read Q, read D,
    write one value per (document, query token) (Sec. 2.3, Eq. (5))."""
    return nq_tok * d * elem + B * nd_tok * d * elem + B * nq_tok * out_bytes


def similarity_bytes(B: int, lq: int, ld: int, elem: int) -> int:
    """Size of the [B, Lq, Ld] similarity tensor the fused kernel never forms."""
    return B * lq * ld * elem


def argmax_bytes(nq: int, nd: int, lq: int) -> int:
    """int32 argmax saved for the backward, [Nq * Nd, Lq]."""
    return nq * nd * lq * 4


def maxsim_flops(q_rows: int, dim: int, d_tokens: int) -> int:
    """Dense contraction FLOPs: 2 * (query rows) * dim * (document tokens)."""
    return 2 * q_rows * dim * d_tokens


def varlen_algorithmic_bytes(nq: int, lq: int, dim: int, total_d: int, nd: int, elem: int = 2) -> int:
    """Bytes one varlen forward must move: Q, packed D, cu_seqlens, scores."""
    return nq * lq * dim * elem + total_d * dim * elem + (nd + 1) * 4 + nq * nd * 4


def shard_documents(lens: np.ndarray, rank: int, world: int):
    """Contiguous documents [j0, j1) of one rank, balanced by token count: the
    first document whose start reaches rank * total / world opens the range."""
    cu = np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))])
    total = int(cu[-1])
    nd = len(cu) - 1

    def first(r):
        if r <= 0:
            return 0
        if r >= world:
            return nd
        return int(np.searchsorted(cu[:-1], (total * r) // world, side="left"))

    return first(rank), first(rank + 1)


# ---------------------------------------------------------------- helpers

def kernel_source_hash(workload: str) -> str:
    """Hash of the device sources of the workload's dominant kernel."""
    files = ("chamfer_kernels.cuh",) if workload.startswith("chamfer") else ("fwd_kernel.cuh", "ptx.cuh")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "maxsim_scoring_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# DRAM traffic (read + write bytes) of the forward kernel per launch on a
# workload's default size, scaled by the document tokens from one ncu capture
# of a smaller instance (the ncu summary of the forward on this workload);
# valid only for the kernel sources whose hash is recorded with it.
MEASURED_TRAFFIC = {
    # (425,491,456 + 3,865,088) B at Nd = 10,000 (1,657,544 tokens), x 16,644,526 / 1,657,544
    ("colbert_varlen", "8c0cc3b61b53f37c"): 4311460908,
    # (270,877,440 + 4,217,600) B at Nd = 2,000 documents of 1,024 tokens, x 10,000 / 2,000
    ("int8_rerank", "8c0cc3b61b53f37c"): 1375475200,
}


def l2_read_gbs(device) -> float:
    """Bandwidth of L2: 20 back-to-back copies between two 24 MiB tensors that
    stay in L2 (129 MB), read plus write bytes, between one pair of CUDA events;
    best of 5."""
    import torch
    x = torch.ones(12 * 1024 * 1024, dtype=torch.bfloat16, device=device)
    y = torch.empty_like(x)
    for _ in range(3):
        y.copy_(x)
    best = 0.0
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(20):
            y.copy_(x)
        e1.record()
        torch.cuda.synchronize(device)
        best = max(best, 20 * 2 * x.numel() * 2 / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return best


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout_s: float = 3.0):
        """Block until the sampler has produced its first reading, so that its
        start-up (driver initialisation) falls before the timed region."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout_s:
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def make_workload(name: str, rank: int, world: int, shard: str, nd: int = 0):
    """Host arrays of a workload for this rank, plus a description."""
    from datagen import workloads
    if name not in workloads.SPECS:
        raise SystemExit(f"unknown workload {name}; one of {sorted(workloads.SPECS)}")
    spec = dict(workloads.SPECS[name])
    if shard == "weak":
        spec["seed"] = spec["seed"] + 1000 * rank  # every rank scores its own documents
    if nd:
        if name.startswith("chamfer"):
            spec["N"] = spec["M"] = nd  # smaller clouds for profiler captures only
        else:
            spec["Nd"] = nd  # smaller instance for profiler captures only
    w = workloads.make(name, **spec)
    w["name"] = name
    if shard == "global" and world > 1:
        if name != "colbert_varlen":
            raise SystemExit("--shard global is implemented for colbert_varlen")
        j0, j1 = shard_documents(w["lens"], rank, world)
        cu = w["cu_seqlens_d"].astype(np.int64)
        w["D"] = np.ascontiguousarray(w["D"][cu[j0]:cu[j1]])
        w["lens"] = w["lens"][j0:j1]
        w["cu_seqlens_d"] = (cu[j0:j1 + 1] - cu[j0]).astype(np.int32)
        w["Nd"], w["total_d"] = j1 - j0, int(cu[j1] - cu[j0])
    return w, spec


def describe(w, spec):
    name = w["name"]
    if name == "chamfer_100k":
        text = (f"chamfer_100k: B={w['B']} pair of point clouds, P [{w['N']},{w['dim']}] and Q [{w['M']},{w['dim']}] "
                f"float32 with N(0,1) coordinates, upstream gradient N(0,1), seed {spec['seed']}; a step is the "
                f"loss forward (nearest points both ways) and the backward through the saved indices")
        cfg = {"workload": text, "B": w["B"], "N": w["N"], "M": w["M"], "dim": w["dim"],
               "l2": "inputs (2.4 MB) stay in L2 by design: the step is bound by the search, not memory; no flush"}
        return cfg
    if name == "colbert_varlen_bwd":
        text = (f"colbert_varlen_bwd: backward of Q [{w['Nq']},{w['Lq']},{w['dim']}] {w['dtype']} vs Nd={w['Nd']} "
                f"packed documents, Ld~U[{spec['ld_min']},{spec['ld_max']}] (sum Ld={w['total_d']}), grad N(0,1), "
                f"argmax from one varlen forward at setup; l2-normalised Gaussian rows, seed {spec['seed']}")
        cfg = {"workload": text, "Nq": w["Nq"], "Lq": w["Lq"], "Nd": w["Nd"], "total_d": w["total_d"], "dim": w["dim"]}
        moved = (w["total_d"] * w["dim"] * 6 + 3 * w["Nq"] * w["Nd"] * w["Lq"] * 4)
        cfg["l2"] = ("D, dD, the argmax and the CSR (%.2f GB) exceed L2: no flush" % (moved / 1e9)
                     if moved > L2_BYTES else "smaller than L2")
        return cfg
    if name == "colpali_out_of_core":
        text = (f"colpali_out_of_core: Q [{w['Nq']},{w['Lq']},{w['dim']}] {w['dtype']} on the device vs a corpus D "
                f"[{w['Nd']},{w['Ld']},{w['dim']}] {w['dtype']} ({w['Nd'] * w['Ld'] * w['dim'] * 2 / 1e9:.1f} GB) in "
                f"page-locked host memory, streamed in blocks of {w['block_docs']} documents; l2-normalised Gaussian "
                f"rows, seed {spec['seed']}")
        cfg = {"workload": text}
        for key in ("Nq", "Lq", "Nd", "Ld", "dim", "block_docs"):
            cfg[key] = w[key]
        cfg["l2"] = "the corpus comes from host memory every step; no flush needed"
        return cfg
    if name == "two_stage_topk":
        text = (f"two_stage_topk: Q [{w['Nq']},{w['Lq']},{w['dim']}] vs D [{w['Nd']},{w['Ld']},{w['dim']}], each as "
                f"INT8 with per-token f32 scales and as f16 (the same l2-normalised Gaussian rows, seed "
                f"{spec['seed']}); stage 1 INT8 scores of every pair, top k1={w['k1']} per query, f16 rescoring of "
                f"the candidates, top k={w['k']}")
        cfg = {"workload": text}
        for key in ("Nq", "Lq", "Nd", "Ld", "dim", "k1", "k"):
            cfg[key] = w[key]
        cfg["l2"] = "inputs larger than L2 (the INT8 corpus alone is %.2f GB); no flush needed" % (
            w["Nd"] * w["Ld"] * (w["dim"] + 4) / 1e9)
        return cfg
    if name == "colbert_varlen":
        text = (f"colbert_varlen: Nq={w['Nq']} queries x Lq={w['Lq']} tokens vs Nd={w['Nd']} packed docs, "
                f"Ld~U[{spec['ld_min']},{spec['ld_max']}] (sum Ld={w['total_d']}), d={w['dim']}, f16, "
                f"l2-normalised Gaussian rows, seed {spec['seed']}")
        d_bytes = w["total_d"] * w["dim"] * 2
    elif name == "colbert_pairs":
        text = (f"colbert_pairs: Nq={w['Nq']} queries x Lq={w['Lq']} tokens, {w['num_pairs']} (query, document) "
                f"pairs ({spec['pairs_per_query']} per query, documents uniform) over Nd={w['Nd']} packed docs, "
                f"Ld~U[{spec['ld_min']},{spec['ld_max']}], d={w['dim']}, f16, l2-normalised Gaussian rows, "
                f"seed {spec['seed']}")
        d_bytes = w["total_d"] * w["dim"] * 2
    elif name == "int8_rerank":
        text = (f"int8_rerank: Q int8 [{w['Nq']},{w['Lq']},{w['dim']}] (query rows in 512-row chunks), "
                f"D int8 [{w['Nd']},{w['Ld']},{w['dim']}], per-token f32 scales of l2-normalised Gaussian rows, "
                f"seed {spec['seed']}")
        d_bytes = w["Nd"] * w["Ld"] * w["dim"]
    else:
        masks = (" q_mask drops the last U{0..40} tokens, d_mask hides U{0..200} random patches;"
                 if name == "colpali_cross" else "")
        text = (f"{name}: Q [{w['Nq']},{w['Lq']},{w['dim']}] vs D [{w['Nd']},{w['Ld']},{w['dim']}] {w['dtype']},"
                f"{masks} l2-normalised Gaussian rows, seed {spec['seed']}")
        d_bytes = w["Nd"] * w["Ld"] * w["dim"] * 2
    cfg = {"workload": text}
    for k in ("Nq", "Lq", "Nd", "Ld", "total_d", "num_pairs", "dim"):
        if k in w:
            cfg[k] = w[k]
    cfg["l2"] = ("inputs larger than L2 (D alone is %.2f GB); no flush needed" % (d_bytes / 1e9)
                 if d_bytes > L2_BYTES else
                 "inputs smaller than L2: a 256 MiB buffer is rewritten before every timed step")
    return cfg


# ---------------------------------------------------------------- the oracle arm

def units_of(w) -> int:
    """Documents scored per step: every (query, document) pair of a pair list;
    for Chamfer, pairs of point clouds."""
    if w["name"].startswith("chamfer"):
        return w["B"]
    return w["num_pairs"] if "num_pairs" in w else w["Nd"]


def time_oracle(w, n_docs: int, threads: int = 0):  # threads 0: all host cores
    """Oracle docs/s on the first n_docs documents (pairs, for a pair list) -
    a bounded sample."""
    import oracle
    docs = np.arange(n_docs, dtype=np.int64)
    t0 = time.perf_counter()
    name = w["name"]
    if name == "colbert_pairs":
        pr = w["pairs"][:n_docs]
        for i in np.unique(pr[:, 0]):
            rows = w["Q"][i].reshape(-1, w["dim"])
            oracle.fwd_packed(rows, np.array([0, w["Lq"]], dtype=np.int64), w["D"],
                              w["cu_seqlens_d"].astype(np.int64), "f16", docs=pr[pr[:, 0] == i, 1].astype(np.int64),
                              threads=threads)
    elif name == "colbert_varlen":
        q_off = np.arange(w["Nq"] + 1, dtype=np.int64) * w["Lq"]
        oracle.fwd_packed(w["Q"].reshape(-1, w["dim"]), q_off, w["D"], w["cu_seqlens_d"].astype(np.int64), "f16",
                          docs=docs, threads=threads)
    elif name == "int8_rerank":
        oracle.fwd_int8(w["Q"], w["q_scale"], w["D"], w["d_scale"], docs=docs, threads=threads)
    elif name == "colpali_out_of_core":
        from datagen import workloads
        D = workloads.fill_corpus(dict(w, Nd=n_docs), np.empty((n_docs * w["Ld"], w["dim"]), np.uint16))
        t0 = time.perf_counter()  # the corpus sample is generated outside the timing
        oracle.fwd_dense(w["Q"], D.reshape(n_docs, w["Ld"], w["dim"]), w["dtype"], threads=threads)
    elif name == "two_stage_topk":
        k1 = min(w["k1"], n_docs)
        oracle.two_stage_topk(w["Q8"], w["q_scale"], w["D8"][:n_docs], w["d_scale"][:n_docs], w["Q16"],
                              w["D16"][:n_docs], "f16", k1, min(w["k"], k1), threads=threads)
    elif name == "contrastive_bwd":
        # the backward needs its forward: argmax of the sampled documents, then dQ, dD and the CSR
        Ds = np.ascontiguousarray(w["D"][:n_docs])
        _, am, _ = oracle.fwd_dense(w["Q"], Ds, w["dtype"], threads=threads)
        oracle.bwd(w["Q"], Ds, w["dtype"], am, np.ascontiguousarray(w["grad"][:, :n_docs]), threads=threads)
    else:
        oracle.fwd_dense(w["Q"], w["D"], w["dtype"], q_mask=w.get("q_mask"), d_mask=w.get("d_mask"), docs=docs,
                         threads=threads)
    dt = time.perf_counter() - t0
    return n_docs / dt, dt


def time_chamfer_oracle(w, k: int):
    """Oracle cloud pairs/s from the first k points of P against all of Q (both
    directions: 2 k M distance evaluations) plus the backward of that pair,
    scaled by the 2 N M evaluations of a full pair."""
    import oracle
    P, Q = w["P"][:, :k], w["Q"]
    t0 = time.perf_counter()
    _, ip, _, _, iq, _, _ = oracle.chamfer_fwd(P, Q)
    oracle.chamfer_bwd(P, Q, ip, iq, w["grad"])
    dt = time.perf_counter() - t0
    frac = (2.0 * k * w["M"]) / (2.0 * w["N"] * w["M"])
    return w["B"] * frac / dt, dt


def calibrated_sample(w, target_s: float):
    if w["name"].startswith("chamfer"):
        probe = 64
        _, dt = time_chamfer_oracle(w, probe)
        return int(max(probe, min(w["N"], probe * target_s / max(dt, 1e-9))))
    probe = min(8, units_of(w))
    rate, _ = time_oracle(w, probe)
    return int(max(probe, min(units_of(w), rate * target_s)))


def oracle_sample(w, n: int, threads: int = 0):
    """(rate, seconds, description) of the oracle on a bounded sample."""
    if w["name"].startswith("chamfer"):
        rate, dt = time_chamfer_oracle(w, n)
        return rate, dt, (f"first {n} of {w['N']} points of P against all {w['M']} of Q, both directions, "
                          f"plus that pair's backward, scaled by the distance evaluations of a full pair")
    rate, dt = time_oracle(w, n, threads)
    what = (f"first {n} of {w['num_pairs']} pairs" if "num_pairs" in w else
            f"first {n} of {w['Nd']} documents, all {w['Nq']} queries")
    if w["name"] == "contrastive_bwd":
        what += " (the forward for their argmax, then dQ, dD and the CSR)"
    return rate, dt, what


def oracle_cores(w) -> int:
    """Threads the oracle actually runs: the Chamfer oracle parallelises over
    the B pairs of clouds only."""
    import oracle
    if w["name"].startswith("chamfer"):
        return max(1, min(oracle.max_threads(), w["B"]))
    return oracle.max_threads()


def run_reference(args, rank, world):
    import oracle
    if rank != 0:
        return
    w, spec = make_workload(args.workload, 0, 1, "weak", args.nd)
    cores = oracle_cores(w)
    metric, unit = metric_of(args.workload)
    n = calibrated_sample(w, target_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, n)
    rates, times = [], []
    for _ in range(args.steps):
        rate, dt, what = oracle_sample(w, n)
        rates.append(rate)
        times.append(dt)
    value = args.steps / sum(1.0 / r for r in rates)
    sample = f"{what}, per step"
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(w, spec),
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm

class Case:
    """One workload on one GPU: device inputs, the timed call, and the bytes /
    FLOPs that bound it."""

    def __init__(self, w, device):
        import torch as t

        from maxsim_scoring_gb300 import _native, ops
        self.w, self.device, self.ops = w, device, ops
        name = w["name"]
        self.name = name

        def pinned_half(bits, dtype):
            return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dtype).pin_memory()

        def pinned(x):
            return t.from_numpy(np.ascontiguousarray(x)).pin_memory()

        self.h_in, self.d_in = {}, {}
        if name == "int8_rerank":
            for k in ("Q", "q_scale", "D", "d_scale"):
                self.h_in[k] = pinned(w[k])
        else:
            dt = t.float16 if w["dtype"] == "f16" else t.bfloat16
            self.h_in["Q"], self.h_in["D"] = pinned_half(w["Q"], dt), pinned_half(w["D"], dt)
            for k in ("cu_seqlens_d", "q_mask", "d_mask", "grad", "pairs"):
                if w.get(k) is not None:
                    self.h_in[k] = pinned(w[k])
        for k, v in self.h_in.items():
            self.d_in[k] = v.to(device)
        self.e2e_in = {k: t.empty_like(v) for k, v in self.d_in.items()}
        Nq, Nd, dim = w["Nq"], w["Nd"], w["dim"]
        out_shape = (w["num_pairs"],) if name == "colbert_pairs" else (Nq, Nd)
        self.scores = t.empty(out_shape, dtype=t.float32, device=device)
        self.h_scores = t.empty(out_shape, dtype=t.float32).pin_memory()
        self.units = units_of(w)
        self.argmax = None
        if name == "colbert_varlen":
            Lq, T = w["Lq"], w["total_d"]
            ws = ops.workspace_size(_native.OP_FWD_VARLEN, Nq, Lq, Nd, T, dim)
            self.flops = maxsim_flops(Nq * Lq, dim, T)
            self.bytes = varlen_algorithmic_bytes(Nq, Lq, dim, T, Nd)
            self.bound, self.dtype, self.launches = "tensor", "f16", 3
        elif name == "colbert_pairs":
            Lq, T, n = w["Lq"], w["total_d"], w["num_pairs"]
            ws = ops.workspace_size(_native.OP_SCORE_PAIRS, Nq, Lq, Nd, n, dim)
            lens = np.diff(w["cu_seqlens_d"].astype(np.int64))
            tokens = int(lens[w["pairs"][:, 1]].sum())  # every pair streams its document
            self.flops = maxsim_flops(Lq, dim, tokens)
            # per pair: its document's rows, the pair, two offsets, the score; plus Q
            self.bytes = tokens * dim * 2 + n * (8 + 8 + 4) + Nq * Lq * dim * 2
            self.bound, self.dtype, self.launches = "hbm", "f16", 6
        elif name == "int8_rerank":
            Lq, Ld = w["Lq"], w["Ld"]
            ws = ops.workspace_size(_native.OP_FWD_INT8, Nq, Lq, Nd, Ld, dim)
            self.flops = maxsim_flops(Nq * Lq, dim, Nd * Ld)
            self.bytes = Nq * Lq * (dim + 4) + Nd * Ld * (dim + 4) + Nq * Nd * 4
            self.bound, self.dtype, self.launches = "tensor", "int8 (f16 MMA, fp32 acc)", 3
        else:
            Lq, Ld = w["Lq"], w["Ld"]
            self.argmax = t.empty((Nq * Nd, Lq), dtype=t.int32, device=device)
            ws = max(ops.workspace_size(_native.OP_FWD, Nq, Lq, Nd, Ld, dim),
                     ops.workspace_size(_native.OP_BWD, Nq, Lq, Nd, Ld, dim))
            self.dtype = w["dtype"]
            if name == "contrastive_bwd":
                ops.maxsim_fwd(self.d_in["Q"], self.d_in["D"], argmax=self.argmax, want_argmax=True)
                self.dQ = t.empty((Nq, Lq, dim), dtype=t.float32, device=device)
                self.dD = t.empty((Nd, Ld, dim), dtype=t.float32, device=device)
                self.flops = 2 * 2 * Nq * Nd * Lq * dim
                # The call asks for no CSR arrays, so the CSR of each document
                # slice stays in shared memory: read Q, D, the argmax and g once,
                # write dQ and dD once. Besides, every source gathers one Q row
                # (dD) and one D row (dQ), served from L2: the secondary bound.
                self.bytes = (Nq * Lq * dim * 2 + Nd * Ld * dim * 2 + Nq * Nd * Lq * 4 + Nq * Nd * 4
                              + (Nq * Lq + Nd * Ld) * dim * 4)
                self.gather_bytes = 2 * Nq * Nd * Lq * dim * 2
                self.bound, self.launches = "hbm", 2
            else:
                self.flops = maxsim_flops(Nq * Lq, dim, Nd * Ld)
                self.bytes = (Nq * Lq * dim * 2 + Nd * Ld * dim * 2 + Nq * Nd * 4 + Nq * Nd * Lq * 4
                              + (Nq * Lq + Nd * Ld if name == "colpali_cross" else 0))
                self.bound = "hbm" if name == "tiny_rerank" else "tensor"
                self.launches = 1
        self.ws = t.empty(max(1, ws), dtype=t.uint8, device=device)
        if name == "colbert_varlen":
            self.h_cu = self.h_in["cu_seqlens_d"]  # page-locked host offsets of the corpus
            self.e2e_ws = t.empty(ops.workspace_size(_native.OP_FWD_VARLEN_STREAMED, Nq, w["Lq"], min(5000, Nd),
                                                     1 << 20, dim), dtype=t.uint8, device=device)
            self.e2e_api = "maxsim_fwd_varlen_streamed (host corpus, 5,000-document blocks)"
        in_bytes = sum(v.numel() * v.element_size() for v in self.d_in.values())
        self.flush_buf = (t.empty(256 * 1024 * 1024 // 4, dtype=t.float32, device=device)
                          if in_bytes < 2 * L2_BYTES else None)

    def call(self, d):
        w, ops, name = self.w, self.ops, self.name
        if name == "colbert_varlen":
            ops.maxsim_fwd_varlen(d["Q"], None, w["Lq"], d["D"], d["cu_seqlens_d"], scores=self.scores,
                                  workspace=self.ws)
        elif name == "colbert_pairs":
            ops.maxsim_score_pairs_packed(d["Q"], None, w["Lq"], d["D"], d["cu_seqlens_d"], d["pairs"],
                                          scores=self.scores, workspace=self.ws)
        elif name == "int8_rerank":
            ops.maxsim_fwd_int8(d["Q"], d["q_scale"], d["D"], d["d_scale"], scores=self.scores, workspace=self.ws)
        elif name == "contrastive_bwd":
            ops.maxsim_bwd(d["Q"], d["D"], self.argmax, d["grad"], dQ=self.dQ, dD=self.dD, workspace=self.ws)
        else:
            ops.maxsim_fwd(d["Q"], d["D"], d.get("q_mask"), d.get("d_mask"), scores=self.scores,
                           argmax=self.argmax, want_argmax=True, workspace=self.ws)

    def step(self):
        self.call(self.d_in)

    def e2e_step(self):
        if self.name == "colbert_varlen":
            # a corpus in host memory goes through the out-of-core call: its
            # document blocks are copied while the previous block is scored
            self.e2e_in["Q"].copy_(self.h_in["Q"], non_blocking=True)
            self.ops.maxsim_fwd_varlen_streamed(self.e2e_in["Q"], None, self.w["Lq"], self.h_in["D"],
                                                self.h_cu, block_docs=5000, block_tokens=1 << 20,
                                                scores=self.scores, workspace=self.e2e_ws)
            self.h_scores.copy_(self.scores, non_blocking=True)
            return
        for k, v in self.h_in.items():
            self.e2e_in[k].copy_(v, non_blocking=True)
        self.call(self.e2e_in)
        if self.name == "contrastive_bwd":
            self.dQ.cpu()  # the step's result comes back to the host
        else:
            self.h_scores.copy_(self.scores, non_blocking=True)

    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.h_in.values())

    def d2h_bytes(self):
        if self.name == "contrastive_bwd":
            return self.dQ.numel() * 4
        return self.scores.numel() * 4

    def flush(self):
        if self.flush_buf is not None:
            self.flush_buf.add_(1.0)


class ChamferCase:
    """Chamfer distance of one pair of 100K-point clouds: a step is the
    forward (nearest points both ways, loss) and the backward through the
    saved indices. The forward call is also timed on its own: its nearest-
    point kernel dominates the step and carries the roofline."""

    def __init__(self, w, device):
        import torch as t

        from maxsim_scoring_gb300 import _native, ops
        self.w, self.device, self.ops, self.t = w, device, ops, t
        self.name = w["name"]
        B, N, M, dim = w["B"], w["N"], w["M"], w["dim"]
        self.h_in = {k: t.from_numpy(np.ascontiguousarray(w[k])).pin_memory() for k in ("P", "Q", "grad")}
        self.d_in = {k: v.to(device) for k, v in self.h_in.items()}
        self.e2e_in = {k: t.empty_like(v) for k, v in self.d_in.items()}
        self.ws_f = t.empty(ops.workspace_size(_native.OP_CHAMFER_FWD, B, N, M, 0, dim), dtype=t.uint8, device=device)
        self.ws_b = t.empty(max(1, ops.workspace_size(_native.OP_CHAMFER_BWD, B, N, M, 0, dim)), dtype=t.uint8,
                            device=device)
        self.dP = t.empty((B, N, dim), dtype=t.float32, device=device)
        self.dQ = t.empty((B, M, dim), dtype=t.float32, device=device)
        self.h_out = {"loss": t.empty(B, dtype=t.float32).pin_memory(),
                      "dP": t.empty((B, N, dim), dtype=t.float32).pin_memory(),
                      "dQ": t.empty((B, M, dim), dtype=t.float32).pin_memory()}
        self.units = B
        self.fma = chamfer_fma(B, N, M, dim)
        self.bytes = (B * (N + M) * dim * 4) * 2 + B * (N + M) * 8
        if dim <= 4:
            # tensor cores: one augmented inner product of 3 dim + 2 tf32 terms per pair
            self.flops = 2 * B * N * M * 2 * (3 * dim + 2)
            self.bound, self.dtype, self.peak_ratio = "tensor", "f32 (two-part tf32 split, fp32 accumulation)", 1.1 / 2.25
        else:
            self.flops = 2 * self.fma
            self.bound, self.dtype, self.peak_ratio = "alu", "f32", None
        K = B * (N + M)
        passes = max(1, -(-int(K).bit_length() // 9))  # 9-bit digits
        # forward: (2 operand preps +) search, merge, loss | backward: keys, radix passes, row_ptr, grad
        self.launches = (5 if dim <= 4 else 3) + 1 + 3 * passes + 2
        self.events = None
        self.loss = None

    def call(self, d):
        ops = self.ops
        stream = self.t.cuda.current_stream(self.device)
        if self.events is not None:
            e0, e1 = self.t.cuda.Event(enable_timing=True), self.t.cuda.Event(enable_timing=True)
            e0.record(stream)
        self.loss, _, ip, _, iq = ops.chamfer_fwd(d["P"], d["Q"], workspace=self.ws_f)
        if self.events is not None:
            e1.record(stream)
            self.events.append((e0, e1))
        ops.chamfer_bwd(d["P"], d["Q"], ip, iq, d["grad"], dP=self.dP, dQ=self.dQ, workspace=self.ws_b)

    def step(self):
        self.call(self.d_in)

    def e2e_step(self):
        for k, v in self.h_in.items():
            self.e2e_in[k].copy_(v, non_blocking=True)
        self.call(self.e2e_in)
        self.h_out["loss"].copy_(self.loss, non_blocking=True)
        self.h_out["dP"].copy_(self.dP, non_blocking=True)
        self.h_out["dQ"].copy_(self.dQ, non_blocking=True)

    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.h_in.values())

    def d2h_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.h_out.values())

    def flush(self):
        pass

    def start_kernel_timing(self):
        self.events = []

    def kernel_ms(self):
        ev, self.events = self.events, None
        return sum(a.elapsed_time(b) for a, b in ev) / max(1, len(ev))


class TwoStageCase:
    """Two-stage INT8 -> f16 top-k over the whole corpus: INT8 scores of every
    (query, document), the k1 best per query, their f16 rescoring, the k best.
    The INT8 forward dominates the step."""

    def __init__(self, w, device):
        import torch as t

        from maxsim_scoring_gb300 import _native, ops
        self.w, self.device, self.ops, self.t = w, device, ops, t
        self.name = w["name"]
        Nq, Lq, Nd, Ld, dim, k1, k = (w[x] for x in ("Nq", "Lq", "Nd", "Ld", "dim", "k1", "k"))

        def pinned(x):
            return t.from_numpy(np.ascontiguousarray(x)).pin_memory()

        self.h_in = {key: pinned(w[key]) for key in ("Q8", "q_scale", "D8", "d_scale")}
        for key in ("Q16", "D16"):
            self.h_in[key] = t.from_numpy(np.ascontiguousarray(w[key]).view(np.int16)).view(t.float16).pin_memory()
        self.d_in = {key: v.to(device) for key, v in self.h_in.items()}
        self.e2e_in = {key: t.empty_like(v) for key, v in self.d_in.items()}
        self.ws = t.empty(ops.workspace_size(_native.OP_TWO_STAGE, Nq, Lq, Nd, Ld, dim), dtype=t.uint8, device=device)
        self.h_out = {"idx": t.empty((Nq, k), dtype=t.int32).pin_memory(),
                      "scores": t.empty((Nq, k), dtype=t.float32).pin_memory()}
        self.out = None
        self.units = Nd
        # stage 1 over the corpus plus stage 2 over Nq * k1 candidates
        self.flops = maxsim_flops(Nq * Lq, dim, Nd * Ld) + maxsim_flops(Lq, dim, Nq * k1 * Ld)
        self.bytes = Nd * Ld * (dim + 4) + Nq * k1 * Ld * dim * 2 + Nq * Nd * 4
        self.bound, self.dtype = "tensor", "int8 then f16 (f16 MMA, fp32 acc)"
        # int8: repack + forward; topk; pairs + offsets; pairs: check_cu, count, scan, place, repack, forward; topk
        self.launches = 2 + 1 + 2 + 6 + 1

    def call(self, d):
        w = self.w
        self.out = self.ops.maxsim_two_stage_topk(d["Q8"], d["q_scale"], d["D8"], d["d_scale"], d["Q16"], d["D16"],
                                                  w["k1"], w["k"], workspace=self.ws)

    def step(self):
        self.call(self.d_in)

    def e2e_step(self):
        for key, v in self.h_in.items():
            self.e2e_in[key].copy_(v, non_blocking=True)
        self.call(self.e2e_in)
        self.h_out["idx"].copy_(self.out[0], non_blocking=True)
        self.h_out["scores"].copy_(self.out[1], non_blocking=True)

    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.h_in.values())

    def d2h_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.h_out.values())

    def flush(self):
        pass  # the corpus (1.7 GB INT8 + 3.3 GB f16) is far larger than L2


class VarlenBwdCase:
    """Backward over packed documents (maxsim_bwd_varlen) through the argmax
    of one varlen forward done at setup: CSR build, dD, dQ."""

    def __init__(self, w, device):
        import torch as t

        from maxsim_scoring_gb300 import _native, ops
        self.w, self.device, self.ops, self.t = w, device, ops, t
        self.name = w["name"]
        Nq, Lq, Nd, T, dim = w["Nq"], w["Lq"], w["Nd"], w["total_d"], w["dim"]
        dt = t.bfloat16 if w["dtype"] == "bf16" else t.float16

        def pinned(x):
            return t.from_numpy(np.ascontiguousarray(x)).pin_memory()

        self.h_in = {"Q": t.from_numpy(np.ascontiguousarray(w["Q"]).view(np.int16)).view(dt).pin_memory(),
                     "D": t.from_numpy(np.ascontiguousarray(w["D"]).view(np.int16)).view(dt).pin_memory(),
                     "cu_seqlens_d": pinned(w["cu_seqlens_d"]), "grad": pinned(w["grad"])}
        self.d_in = {k: v.to(device) for k, v in self.h_in.items()}
        self.e2e_in = {k: t.empty_like(v) for k, v in self.d_in.items()}
        _, self.argmax = ops.maxsim_fwd_varlen(self.d_in["Q"], None, Lq, self.d_in["D"], self.d_in["cu_seqlens_d"],
                                               want_argmax=True)
        self.h_argmax = self.argmax.cpu().pin_memory()
        self.h_in["argmax"] = self.h_argmax
        self.d_in["argmax"] = self.argmax
        self.e2e_in["argmax"] = t.empty_like(self.argmax)
        self.ws = t.empty(ops.workspace_size(_native.OP_BWD_VARLEN, Nq, Lq, Nd, T, dim), dtype=t.uint8, device=device)
        self.out = None
        self.h_dq = t.empty((Nq, Lq, dim), dtype=t.float32).pin_memory()
        self.units = Nd
        n_src = Nq * Nd * Lq
        self.flops = 2 * 2 * Nq * Nd * Lq * dim
        # read Q, D, argmax (count and place), g; write and re-read the CSR; write dQ and dD
        self.bytes = (Nq * Lq * dim * 2 + T * dim * 2 + 2 * n_src * 4 + Nq * Nd * 4
                      + 2 * (T + 1 + n_src) * 4 + (Nq * Lq + T) * dim * 4)
        self.bound, self.dtype, self.launches = "hbm", w["dtype"], 6  # check_cu, count, scan, build, dD, dQ

    def call(self, d):
        w = self.w
        self.out = self.ops.maxsim_bwd_varlen(d["Q"], None, w["Lq"], d["D"], d["cu_seqlens_d"], w["max_ld"],
                                              d["argmax"], d["grad"], workspace=self.ws)

    def step(self):
        self.call(self.d_in)

    def e2e_step(self):
        for k, v in self.h_in.items():
            self.e2e_in[k].copy_(v, non_blocking=True)
        self.call(self.e2e_in)
        self.h_dq.copy_(self.out[0], non_blocking=True)

    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.h_in.values())

    def d2h_bytes(self):
        return self.h_dq.numel() * 4

    def flush(self):
        pass  # D (0.17 GB), argmax and the CSR exceed L2 together; see config


class OutOfCoreCase:
    """One query against a corpus in page-locked host memory, scored block by
    block (maxsim_fwd_streamed). The host-to-device link bounds it: its peak
    is a plain pinned copy measured here."""

    def __init__(self, w, device):
        import torch as t

        from datagen import workloads
        from maxsim_scoring_gb300 import _native, ops
        self.w, self.device, self.ops, self.t = w, device, ops, t
        self.name = w["name"]
        Nq, Lq, Nd, Ld, dim, blk = (w[x] for x in ("Nq", "Lq", "Nd", "Ld", "dim", "block_docs"))
        dt = t.bfloat16 if w["dtype"] == "bf16" else t.float16
        self.h_q = t.from_numpy(np.ascontiguousarray(w["Q"]).view(np.int16)).view(dt).pin_memory()
        self.d_q = self.h_q.to(device)
        self.e2e_q = t.empty_like(self.d_q)
        corpus = t.empty((Nd * Ld, dim), dtype=t.int16).pin_memory()
        workloads.fill_corpus(w, corpus.numpy().view(np.uint16))
        self.D_host = corpus.view(dt).view(Nd, Ld, dim)
        self.scores = t.empty((Nq, Nd), dtype=t.float32, device=device)
        self.h_scores = t.empty((Nq, Nd), dtype=t.float32).pin_memory()
        self.ws = t.empty(ops.workspace_size(_native.OP_FWD_STREAMED, Nq, Lq, min(blk, Nd), Ld, dim), dtype=t.uint8,
                          device=device)
        self.units = Nd
        self.corpus_bytes = Nd * Ld * dim * 2
        self.bytes = self.corpus_bytes + Nq * Lq * dim * 2 + Nq * Nd * 4
        self.flops = maxsim_flops(Nq * Lq, dim, Nd * Ld)
        self.bound, self.dtype = "h2d", w["dtype"]
        n_blocks = -(-Nd // blk)
        self.launches = n_blocks * (1 + (0 if Lq % 32 == 0 else 1))  # forward (+ query repack) per block
        self.peak_gbs = self._copy_peak()

    def _copy_peak(self):
        """GB/s of one plain cudaMemcpyAsync of 4 GiB of the pinned corpus."""
        t = self.t
        n = min(self.corpus_bytes, 4 << 30) // 2
        src = self.D_host.view(-1)[:n]
        dst = t.empty(n, dtype=src.dtype, device=self.device)
        best = 0.0
        for _ in range(3):
            e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
            e0.record()
            dst.copy_(src, non_blocking=True)
            e1.record()
            t.cuda.synchronize(self.device)
            best = max(best, 2 * n / (e0.elapsed_time(e1) / 1e3) / 1e9)
        del dst
        return best

    def call(self, q):
        self.ops.maxsim_fwd_streamed(q, self.D_host, block_docs=self.w["block_docs"], scores=self.scores,
                                     workspace=self.ws)

    def step(self):
        self.call(self.d_q)

    def e2e_step(self):
        self.e2e_q.copy_(self.h_q, non_blocking=True)
        self.call(self.e2e_q)
        self.h_scores.copy_(self.scores, non_blocking=True)

    def h2d_bytes(self):
        return self.corpus_bytes + self.h_q.numel() * 2

    def d2h_bytes(self):
        return self.h_scores.numel() * 4

    def flush(self):
        pass  # the corpus arrives from host memory every step


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from maxsim_scoring_gb300 import _native, ops

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    _native.lib()  # fail loudly without the extension
    w, spec = make_workload(args.workload, rank, world, args.shard, args.nd)
    case = (ChamferCase(w, device) if args.workload.startswith("chamfer") else
            TwoStageCase(w, device) if args.workload == "two_stage_topk" else
            OutOfCoreCase(w, device) if args.workload == "colpali_out_of_core" else
            VarlenBwdCase(w, device) if args.workload == "colbert_varlen_bwd" else Case(w, device))
    metric, unit_name = metric_of(args.workload)
    stream = torch.cuda.current_stream(device)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        case.flush()
        case.step()
    torch.cuda.synchronize(device)
    if ops.device_status(device) != 0:
        raise SystemExit("device status after warm-up is not OK")

    clocks = ClockSampler(local_rank)
    clocks.start()
    clocks.wait_first()
    barrier()
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if hasattr(case, "start_kernel_timing"):
        case.start_kernel_timing()
    for k in range(args.steps):
        case.flush()  # outside the events (no-op for inputs larger than L2)
        starts[k].record(stream)
        case.step()
        ends[k].record(stream)
    torch.cuda.synchronize(device)
    barrier()
    clk = clocks.stop()
    per_step_ms = [starts[k].elapsed_time(ends[k]) for k in range(args.steps)]
    total_ms = sum(per_step_ms)
    kernel_ms = case.kernel_ms() if hasattr(case, "kernel_ms") else None
    if ops.device_status(device) != 0:
        raise SystemExit("device status after the timed steps is not OK")

    # end to end through the same public call: H2D of the step's inputs, the
    # call, D2H of the result, all on the stream and inside the events
    # per-step events; the host-to-device link of these machines is shared and
    # has slow episodes, so the line reports the median step (the mean too)
    e2e_steps = max(1, args.steps)
    barrier()
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(e2e_steps)]
    for k in range(e2e_steps):
        ev[k][0].record(stream)
        case.e2e_step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    barrier()
    e2e_each = [a.elapsed_time(b) for a, b in ev]
    e2e_ms = statistics.median(e2e_each)
    e2e_mean_ms = sum(e2e_each) / len(e2e_each)

    # A call this small is sized by its launch: also time many calls back to
    # back (inputs stay in L2 between them; host launch overhead included)
    amortized = None
    if case.name == "tiny_rerank":
        reps = 200
        torch.cuda.synchronize(device)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            case.step()
        a1.record(stream)
        torch.cuda.synchronize(device)
        per_call = a0.elapsed_time(a1) / reps
        amortized = {"calls": reps, "ms_per_call": per_call, "value": case.units / (per_call / 1e3),
                     "unit": unit_name, "note": "back-to-back calls, no L2 flush between them"}

    # max over ranks; units summed over ranks
    t = torch.tensor([total_ms, e2e_ms], dtype=torch.float64, device=device)
    units = torch.tensor([case.units], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(units, op=dist.ReduceOp.SUM)
    total_ms, e2e_ms, all_units = float(t[0]), float(t[1]), float(units[0])
    if rank != 0:
        return

    ms = total_ms / args.steps
    value = all_units / (ms / 1e3)
    peaks, peak_src = load_peaks()
    if case.bound == "h2d":
        achieved = case.corpus_bytes / (ms / 1e3) / 1e9
        peak, unit = round(case.peak_gbs, 1), "GB/s"
        src = "host-to-device link: a plain 4 GiB pinned cudaMemcpyAsync measured in this run"
    elif case.bound == "alu":
        # fp32 FMA peak: lanes x SMs x 2 FLOP x the maximum SM clock
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        max_mhz = clk.get("sm_max_mhz") or 2070.0
        peak = round(FP32_LANES_PER_SM * sms * 2 * max_mhz * 1e6 / 1e12, 2)
        achieved = case.flops / (kernel_ms / 1e3) / 1e12
        unit = "TFLOP/s"
        src = (f"fp32 FMA peak derived from {FP32_LANES_PER_SM} lanes/SM x {sms} SMs x 2 FLOP x {max_mhz:.0f} MHz "
               f"(maximum SM clock)")
    elif case.bound == "tensor":
        kms = kernel_ms if kernel_ms is not None else ms
        achieved = case.flops / (kms / 1e3) / 1e12
        sustained = total_ms > 1000.0
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        unit = "TFLOP/s"
        src = f"{peak_src} {'sustained' if sustained else 'burst'} dense bf16 (f16 runs at the same rate)"
        ratio = getattr(case, "peak_ratio", None)
        if ratio:
            peak = round(peak * ratio, 1)
            src += " x 1.1/2.25 (the nominal tf32 / bf16 dense ratio): tf32"
    else:
        achieved = case.bytes / (ms / 1e3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
        src = f"{peak_src} HBM copy bandwidth"
    l2_gather = None
    if getattr(case, "gather_bytes", None):
        l2 = l2_read_gbs(device)
        # the step cannot beat moving its HBM bytes at the HBM peak plus its row
        # gathers at the L2 figure (a lower bound of L2, so this bound is optimistic)
        bound_ms = 1e3 * (case.bytes / (peaks["hbm_gbs"] * 1e9) + case.gather_bytes / (l2 * 1e9))
        l2_gather = {"bytes_per_launch": case.gather_bytes,
                     "achieved_gbs": round(case.gather_bytes / (ms / 1e3) / 1e9, 1),
                     "l2_read_gbs": round(l2, 1), "frac": round(case.gather_bytes / (ms / 1e3) / 1e9 / l2, 4),
                     "hbm_plus_l2_bound_ms": round(bound_ms, 5), "frac_hbm_plus_l2": round(bound_ms / ms, 4),
                     "peak_source": "L2 bandwidth measured in this run: 20 back-to-back copies between two "
                                    "24 MiB L2-resident tensors (read + write bytes), best of 5; a "
                                    "streaming copy, so a lower bound of what L2 serves"}
    # Beside the measured denominators: the vendor's nominal dense figures, and
    # for the tensor pipe the per-clock rate (an M = 128, N = 128, K = 16 f16 MMA
    # every 64 cycles: 8,192 FLOP per cycle per SM) at the SM clock sampled under load.
    nominal = {}
    if case.bound == "tensor":
        ratio = getattr(case, "peak_ratio", None) or 1.0
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        mhz = clk.get("sm_mhz") or 2070.0
        nominal = {"peak_nominal": round(NOMINAL_BF16_TFLOPS * ratio, 1),
                   "frac_nominal": round(achieved / (NOMINAL_BF16_TFLOPS * ratio), 4),
                   "peak_at_clock": round(TENSOR_FLOP_PER_CYCLE_SM * ratio * sms * mhz * 1e6 / 1e12, 1),
                   "frac_at_clock": round(achieved / (TENSOR_FLOP_PER_CYCLE_SM * ratio * sms * mhz * 1e6 / 1e12), 4),
                   "nominal_source": f"{NOMINAL_BF16_TFLOPS:.0f} TFLOP/s dense bf16 (vendor figure)"
                                     + (" x 1.1/2.25 for tf32" if ratio != 1.0 else "")
                                     + f"; per-clock: {TENSOR_FLOP_PER_CYCLE_SM} FLOP/cycle/SM x {sms} SMs x "
                                       f"{mhz:.0f} MHz (median SM clock in the timed region)"}
    elif case.bound == "hbm":
        nominal = {"peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                   "nominal_source": f"{NOMINAL_HBM_GBS:.0f} GB/s HBM3e (vendor figure)"}
    traffic = MEASURED_TRAFFIC.get((case.name, kernel_source_hash(case.name))) if not args.nd and world == 1 else None
    roofline = {
        "bound": case.bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
        "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": src, **nominal,
        "kernel": ("backward kernels (whole maxsim_bwd_varlen call)" if case.name == "colbert_varlen_bwd" else
                   "the streamed corpus copy (cudaMemcpyAsync, overlapped with maxsim_fwd_kernel on each block; "
                   "duration = the whole maxsim_fwd_streamed call)" if case.bound == "h2d" else
                   ("chamfer_tc_kernel" if case.bound == "tensor" else "chamfer_nn_kernel") +
                   " (duration = the whole maxsim_chamfer_fwd call, CUDA events per step: "
                   f"{kernel_ms:.4f} ms; it also runs the operand preparation, merge and loss kernels)"
                   if case.name.startswith("chamfer") else
                   "maxsim_fwd_kernel (duration = whole entry-point call, which also runs small helper kernels)"
                   if case.name != "contrastive_bwd" else "backward kernels (whole maxsim_bwd call)"),
        "algorithmic_flops_per_launch": case.flops,
        "algorithmic_bytes_per_launch": case.bytes,
        **({"l2_gather": l2_gather} if l2_gather else {}),
    }
    line = {
        "metric": metric, "value": value, "unit": unit_name, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "strong" if args.shard == "global" else "weak",
        "vs_baseline": None, "dtype": case.dtype, "data": "synthetic", "config": describe(w, spec), "clocks": clk,
        "roofline": roofline,
        "e2e": {"value": all_units / (e2e_ms / 1e3), "unit": unit_name, "h2d_bytes_per_step": case.h2d_bytes(),
                "d2h_bytes_per_step": case.d2h_bytes(), "steps": e2e_steps, "statistic": "median step",
                "value_mean": all_units / (e2e_mean_ms / 1e3) if world == 1 else None,
                "api": getattr(case, "e2e_api", "the same call, inputs copied from page-locked host memory first")},
        "gpu_launches": case.launches * args.steps,
        **({"amortized": amortized} if amortized else {}),
        "step_ms_min_median_max": [min(per_step_ms), statistics.median(per_step_ms), max(per_step_ms)],
    }
    if unit_name == UNIT and "Nq" in w and case.name != "colbert_pairs":  # the pair list counts pairs already
        # every document is scored against every query of the call: (query, document) pairs/s
        line["pairs_per_s"] = value * w["Nq"]
    if world == 1 and not args.no_cpu_baseline and case.name != "colbert_varlen_bwd":
        n = calibrated_sample(w, target_s=args.cpu_seconds)
        rate, dt, what = oracle_sample(w, n)
        line["cpu_baseline"] = {"value": rate, "unit": unit_name, "cores": oracle_cores(w), "kind": "oracle",
                                "sample": f"{what} ({dt:.1f} s)"}
        # the same oracle on one host core, on a sample sized for a few seconds
        cores = oracle_cores(w)
        if cores > 1:
            n1 = max(1, min(n, int(n * args.cpu_seconds / 4.0 / max(dt * cores, 1e-9))))
            rate1, dt1, what1 = oracle_sample(w, n1, threads=1)
            line["cpu_baseline"]["one_core"] = {"value": rate1, "unit": unit_name, "cores": 1,
                                                "sample": f"{what1} ({dt1:.1f} s)"}
        else:
            line["cpu_baseline"]["one_core"] = {"value": rate, "unit": unit_name, "cores": 1,
                                                "sample": "the run above (it uses one core)"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="colbert_varlen")
    ap.add_argument("--shard", choices=["weak", "global"], default="weak")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--nd", type=int, default=0,
                    help="override the document count, or the cloud size for Chamfer (profiler captures only)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
