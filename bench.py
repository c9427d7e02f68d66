#!/usr/bin/env python3
"""MaxSim throughput on one GB300 (docs scored / s) with its roofline.

Default workload: ColBERT rerank over packed documents -- Nq = 32 queries of
Lq = 32 tokens, Nd = 100,000 documents with lengths uniform in [32, 300],
dim = 128, f16, l2-normalised Gaussian rows (seeded, synthetic). A step is one
maxsim_fwd_varlen call scoring every document against every query.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Prints one JSON line (rank 0). Under torchrun every rank scores its own
100,000 documents (weak scaling, no data-path communication); timing is the
maximum over ranks between barriers.

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


# ---------------------------------------------------------------- helpers

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("fwd_kernel.cuh", "ptx.cuh", "maxsim_api.cu"):
        with open(os.path.join(ROOT, "maxsim_scoring_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# DRAM traffic of the forward kernel per launch on this workload, from one ncu
# capture (profiles/maxsim_fwd_kernel__colbert_varlen.md), valid only for the
# kernel sources whose hash is recorded with it.
MEASURED_TRAFFIC = {}


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

def build_workload(name: str, rank: int, nd: int = 0):
    from datagen import workloads
    if name != "colbert_varlen":
        raise SystemExit(f"unknown bench workload {name}")
    spec = dict(workloads.SPECS[name])
    spec["seed"] = spec["seed"] + 1000 * rank  # every rank scores its own documents
    if nd:
        spec["Nd"] = nd  # smaller instance for profiler captures only
    return workloads.varlen(**spec), spec


def describe(w, spec):
    return {
        "workload": (f"colbert_varlen: Nq={w['Nq']} queries x Lq={w['Lq']} tokens vs Nd={w['Nd']} packed docs, "
                     f"Ld~U[{spec['ld_min']},{spec['ld_max']}] (sum Ld={w['total_d']}), d={w['dim']}, f16, "
                     f"l2-normalised Gaussian rows, seed {spec['seed']}"),
        "Nq": w["Nq"], "Lq": w["Lq"], "Nd": w["Nd"], "total_d": w["total_d"], "dim": w["dim"],
        "l2": "inputs larger than L2 (D alone is %.2f GB); no flush needed" % (w["total_d"] * w["dim"] * 2 / 1e9),
    }


# ---------------------------------------------------------------- the oracle arm

def time_oracle(w, n_docs: int, threads: int = 0):
    """Oracle docs/s on the first n_docs documents (a bounded sample)."""
    import oracle
    q_off = np.arange(w["Nq"] + 1, dtype=np.int64) * w["Lq"]
    cu = w["cu_seqlens_d"].astype(np.int64)
    docs = np.arange(n_docs, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.fwd_packed(w["Q"].reshape(-1, w["dim"]), q_off, w["D"], cu, "f16", docs=docs, threads=threads)
    dt = time.perf_counter() - t0
    return n_docs / dt, dt


def calibrated_sample(w, target_s: float):
    rate, _ = time_oracle(w, 32)
    n = int(max(32, min(w["Nd"], rate * target_s)))
    return n


def run_reference(args, rank, world):
    import oracle
    if rank != 0:
        return
    w, spec = build_workload(args.workload, 0, args.nd)
    cores = oracle.max_threads()
    n = calibrated_sample(w, target_s=max(2.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(w, n)
    rates, times = [], []
    for _ in range(args.steps):
        r, dt = time_oracle(w, n)
        rates.append(r)
        times.append(dt)
    value = n * args.steps / sum(times)
    sample = f"first {n} of {w['Nd']} documents per step, all {w['Nq']} queries"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(w, spec),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from maxsim_scoring_gb300 import _native, ops

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    _native.lib()  # fail loudly without the extension
    w, spec = build_workload(args.workload, rank, args.nd)
    Nq, Lq, Nd, dim, total_d = w["Nq"], w["Lq"], w["Nd"], w["dim"], w["total_d"]

    # pinned host copies (the e2e leg copies them in every step)
    h_Q = torch.from_numpy(w["Q"].view(np.int16)).view(torch.float16).pin_memory()
    h_D = torch.from_numpy(w["D"].view(np.int16)).view(torch.float16).pin_memory()
    h_cu = torch.from_numpy(w["cu_seqlens_d"]).pin_memory()
    h_scores = torch.empty((Nq, Nd), dtype=torch.float32).pin_memory()
    Q, D, cu = h_Q.to(device), h_D.to(device), h_cu.to(device)
    scores = torch.empty((Nq, Nd), dtype=torch.float32, device=device)
    ws_bytes = ops.workspace_size(_native.OP_FWD_VARLEN, Nq, Lq, Nd, total_d, dim)
    ws = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        ops.maxsim_fwd_varlen(Q, None, Lq, D, cu, scores=scores, workspace=ws)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    if ops.device_status(device) != 0:
        raise SystemExit("device status after warm-up is not OK")

    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for k in range(args.steps):
        step()
        ev[k + 1].record(stream)
    torch.cuda.synchronize(device)
    barrier()
    clk = clocks.stop()
    per_step_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[args.steps])
    if ops.device_status(device) != 0:
        raise SystemExit("device status after the timed steps is not OK")

    # end to end through the same public call: H2D of the step's inputs, the
    # call, D2H of the scores, all on the stream and inside the events
    e2e_steps = max(1, min(args.steps, 5))
    d_Q, d_D, d_cu = torch.empty_like(Q), torch.empty_like(D), torch.empty_like(cu)
    h2d = h_Q.numel() * 2 + h_D.numel() * 2 + h_cu.numel() * 4
    d2h = Nq * Nd * 4
    barrier()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        d_Q.copy_(h_Q, non_blocking=True)
        d_D.copy_(h_D, non_blocking=True)
        d_cu.copy_(h_cu, non_blocking=True)
        ops.maxsim_fwd_varlen(d_Q, None, Lq, d_D, d_cu, scores=scores, workspace=ws)
        h_scores.copy_(scores, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    # max over ranks
    t = torch.tensor([total_ms, e2e_ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms, e2e_ms = float(t[0]), float(t[1])
    if rank != 0:
        return

    ms = total_ms / args.steps
    value = world * Nd / (ms / 1e3)
    peaks, peak_src = load_peaks()
    flops = maxsim_flops(Nq * Lq, dim, total_d)
    achieved_tflops = flops / (ms / 1e3) / 1e12
    sustained = total_ms > 1000.0
    peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    traffic = MEASURED_TRAFFIC.get(kernel_source_hash())
    roofline = {
        "bound": "tensor", "achieved": round(achieved_tflops, 2), "peak": peak, "unit": "TFLOP/s",
        "frac": round(achieved_tflops / peak, 4), "traffic": traffic,
        "peak_source": f"{peak_src} {'sustained' if sustained else 'burst'} dense bf16 (f16 runs at the same rate)",
        "kernel": "maxsim_fwd_kernel (duration = whole entry-point call incl. two small helper kernels)",
        "algorithmic_flops_per_launch": flops,
        "algorithmic_bytes_per_launch": varlen_algorithmic_bytes(Nq, Lq, dim, total_d, Nd),
    }
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic", "config": describe(w, spec), "clocks": clk, "roofline": roofline,
        "e2e": {"value": world * Nd / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * args.steps,
        "step_ms_min_median_max": [min(per_step_ms), statistics.median(per_step_ms), max(per_step_ms)],
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        n = calibrated_sample(w, target_s=args.cpu_seconds)
        rate, dt = time_oracle(w, n)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                                "sample": f"first {n} of {Nd} documents, all {Nq} queries ({dt:.1f} s)"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="colbert_varlen")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--nd", type=int, default=0, help="override the document count (profiler captures only)")
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
