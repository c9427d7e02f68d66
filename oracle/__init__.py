"""CPU oracle for the MaxSim operator -- TEST INFRASTRUCTURE ONLY.

A plain, slow, double-precision restatement of the operator (``maxsim_oracle.c``)
with a numpy-facing ctypes wrapper. Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package; the CUDA library never
calls it and shares no code with it.

Functions
  fwd_packed / fwd_dense : scores, argmax (lowest index, -1 if no valid token)
                           and the top-2 gap of every query row
  fwd_int8               : INT8 x INT8 scores with per-token scales, argmax,
                           and the int32 dot product at the argmax
  csr                    : inverse-argmax CSR (row_ptr, col)
  bwd                    : dQ, dD through the saved argmax (+ the CSR)
  chamfer_fwd / _bwd     : Chamfer distance of point sets and its gradient
  topk                   : the k largest values of every row (descending,
                           lower index first among equal values)
  two_stage_topk         : INT8 scores over the whole corpus, top-k1
                           candidates, f16 / bf16 rescoring, top-k
See the C source for the page sections each one follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "maxsim_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f16": 0, "bf16": 1, "f64": 2}


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2 -ffp-contract=off -fopenmp) next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        # no fused multiply-add contraction: the same rounding on every host
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC,
                               "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.oracle_fwd.argtypes = [vp, vp, ci, i64, vp, i64, vp, i64, vp, vp, vp, i64, vp, vp, vp, i64, ci]
            lib.oracle_fwd_int8.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp, vp, i64, vp, vp, vp,
                                            vp, ci]
            lib.oracle_csr.argtypes = [vp, i64, i64, i64, i64, vp, vp]
            lib.oracle_bwd.argtypes = [vp, vp, ci, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, ci]
            lib.oracle_chamfer_fwd.argtypes = [vp, vp, i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, ci]
            lib.oracle_chamfer_bwd.argtypes = [vp, vp, i64, i64, i64, i64, vp, vp, vp, vp, vp]
            for f in (lib.oracle_fwd, lib.oracle_fwd_int8, lib.oracle_csr, lib.oracle_bwd, lib.oracle_max_threads,
                      lib.oracle_chamfer_fwd, lib.oracle_chamfer_bwd):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _check_dtype(x, dtype):
    want = np.float64 if dtype == "f64" else np.uint16
    assert x.dtype == want, f"{dtype} inputs are passed as {want.__name__}"


def fwd_packed(Q, q_off, D, d_off, dtype, q_mask=None, d_mask=None, docs=None, lq_stride=None, threads=0):
    """MaxSim over packed rows.

    Q [total_q, dim], D [total_d, dim] (uint16 bits for f16/bf16, float64 for f64);
    q_off [Nq+1], d_off [Nd+1] row offsets; masks one byte per packed row.
    docs: optional subset of document indices to score.
    Returns (scores [Nq, n_sel] f64, argmax [Nq*n_sel, lq_stride] i32, gap f64).
    """
    _check_dtype(Q, dtype)
    _check_dtype(D, dtype)
    dim = Q.shape[-1]
    assert D.shape[-1] == dim
    q_off = np.ascontiguousarray(q_off, dtype=np.int64)
    d_off = np.ascontiguousarray(d_off, dtype=np.int64)
    Nq, Nd = len(q_off) - 1, len(d_off) - 1
    docs_arr = None if docs is None else np.ascontiguousarray(docs, dtype=np.int64)
    n_sel = Nd if docs_arr is None else len(docs_arr)
    if lq_stride is None:
        lq_stride = int(np.max(np.diff(q_off))) if Nq else 0
    scores = np.zeros((Nq, n_sel), dtype=np.float64)
    argmax = np.zeros((Nq * n_sel, lq_stride), dtype=np.int32)
    gap = np.zeros((Nq * n_sel, lq_stride), dtype=np.float64)
    qm = None if q_mask is None else np.ascontiguousarray(q_mask, dtype=np.uint8).reshape(-1)
    dm = None if d_mask is None else np.ascontiguousarray(d_mask, dtype=np.uint8).reshape(-1)
    Qc, Dc = np.ascontiguousarray(Q), np.ascontiguousarray(D)
    rc = _load().oracle_fwd(_p(Qc), _p(Dc), DTYPES[dtype], Nq, _p(q_off), Nd, _p(d_off), dim, _p(qm), _p(dm),
                            _p(docs_arr), n_sel, _p(scores), _p(argmax), _p(gap), lq_stride, threads)
    if rc:
        raise ValueError(f"oracle_fwd failed ({rc})")
    return scores, argmax, gap


def fwd_dense(Q, D, dtype, q_mask=None, d_mask=None, docs=None, threads=0):
    """MaxSim for dense Q [Nq,Lq,dim], D [Nd,Ld,dim]; masks [Nq,Lq] / [Nd,Ld]."""
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    q_off = np.arange(Nq + 1, dtype=np.int64) * Lq
    d_off = np.arange(Nd + 1, dtype=np.int64) * Ld
    return fwd_packed(Q.reshape(Nq * Lq, dim), q_off, D.reshape(Nd * Ld, dim), d_off, dtype, q_mask, d_mask,
                      docs, lq_stride=Lq, threads=threads)


def fwd_int8(Q, q_scale, D, d_scale, q_mask=None, d_mask=None, docs=None, threads=0):
    """INT8 x INT8 MaxSim. Q int8 [Nq,Lq,dim], D int8 [Nd,Ld,dim], scales f32 per token.

    Returns (scores f64 [Nq, n_sel], argmax, win_dot int32, gap).
    """
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    docs_arr = None if docs is None else np.ascontiguousarray(docs, dtype=np.int64)
    n_sel = Nd if docs_arr is None else len(docs_arr)
    scores = np.zeros((Nq, n_sel), dtype=np.float64)
    argmax = np.zeros((Nq * n_sel, Lq), dtype=np.int32)
    win = np.zeros((Nq * n_sel, Lq), dtype=np.int32)
    gap = np.zeros((Nq * n_sel, Lq), dtype=np.float64)
    qm = None if q_mask is None else np.ascontiguousarray(q_mask, dtype=np.uint8)
    dm = None if d_mask is None else np.ascontiguousarray(d_mask, dtype=np.uint8)
    args = [np.ascontiguousarray(a) for a in (Q, q_scale.astype(np.float32), D, d_scale.astype(np.float32))]
    rc = _load().oracle_fwd_int8(_p(args[0]), _p(args[1]), _p(args[2]), _p(args[3]), Nq, Lq, Nd, Ld, dim, _p(qm),
                                 _p(dm), _p(docs_arr), n_sel, _p(scores), _p(argmax), _p(win), _p(gap), threads)
    if rc == 2:
        raise OverflowError("an INT8 dot product does not fit int32")
    if rc:
        raise ValueError(f"oracle_fwd_int8 failed ({rc})")
    return scores, argmax, win, gap


def csr(argmax, Nq, Lq, Nd, Ld):
    """Inverse-argmax CSR: (row_ptr [Nd*Ld+1], col [#non-sentinel sources])."""
    a = np.ascontiguousarray(argmax, dtype=np.int32).reshape(-1)
    assert a.size == Nq * Nd * Lq
    row_ptr = np.zeros(Nd * Ld + 1, dtype=np.int32)
    col = np.zeros(max(1, a.size), dtype=np.int32)
    rc = _load().oracle_csr(_p(a), Nq, Lq, Nd, Ld, _p(row_ptr), _p(col))
    if rc == 3:
        raise ValueError("argmax outside [-1, Ld)")
    if rc:
        raise ValueError(f"oracle_csr failed ({rc})")
    return row_ptr, col[: row_ptr[-1]].copy()


def bwd(Q, D, dtype, argmax, grad, q_mask=None, threads=0):
    """dQ [Nq,Lq,dim], dD [Nd,Ld,dim] (float64) and the CSR, for dense Q / D."""
    _check_dtype(Q, dtype)
    _check_dtype(D, dtype)
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    a = np.ascontiguousarray(argmax, dtype=np.int32).reshape(-1)
    g = np.ascontiguousarray(grad, dtype=np.float32).reshape(-1)
    assert g.size == Nq * Nd
    dQ = np.zeros((Nq, Lq, dim), dtype=np.float64)
    dD = np.zeros((Nd, Ld, dim), dtype=np.float64)
    row_ptr = np.zeros(Nd * Ld + 1, dtype=np.int32)
    col = np.zeros(max(1, a.size), dtype=np.int32)
    qm = None if q_mask is None else np.ascontiguousarray(q_mask, dtype=np.uint8)
    Qc, Dc = np.ascontiguousarray(Q), np.ascontiguousarray(D)
    rc = _load().oracle_bwd(_p(Qc), _p(Dc), DTYPES[dtype], Nq, Lq, Nd, Ld, dim, _p(qm), _p(a), _p(g), _p(dQ),
                            _p(dD), _p(row_ptr), _p(col), threads)
    if rc == 3:
        raise ValueError("argmax outside [-1, Ld)")
    if rc:
        raise ValueError(f"oracle_bwd failed ({rc})")
    return dQ, dD, row_ptr, col[: row_ptr[-1]].copy()


def chamfer_fwd(P, Q, threads=0):
    """Chamfer distance (Sec. 4.2.4) of B pairs of point sets P [B, N, dim],
    Q [B, M, dim] (float32). Returns (dist_p [B,N], idx_p [B,N], gap_p [B,N],
    dist_q [B,M], idx_q [B,M], gap_q [B,M], loss [B]), distances in float64."""
    P = np.ascontiguousarray(P, dtype=np.float32)
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    B, N, dim = P.shape
    M = Q.shape[1]
    assert Q.shape[0] == B and Q.shape[2] == dim
    dp, gp = np.zeros((B, N)), np.zeros((B, N))
    dq, gq = np.zeros((B, M)), np.zeros((B, M))
    ip = np.zeros((B, N), dtype=np.int32)
    iq = np.zeros((B, M), dtype=np.int32)
    loss = np.zeros(B)
    rc = _load().oracle_chamfer_fwd(_p(P), _p(Q), B, N, M, dim, _p(dp), _p(ip), _p(gp), _p(dq), _p(iq), _p(gq),
                                    _p(loss), threads)
    if rc:
        raise ValueError(f"oracle_chamfer_fwd failed ({rc})")
    return dp, ip, gp, dq, iq, gq, loss


def chamfer_bwd(P, Q, idx_p, idx_q, grad):
    """dP [B,N,dim], dQ [B,M,dim] (float64) of sum_b grad[b] * CD(P_b, Q_b)."""
    P = np.ascontiguousarray(P, dtype=np.float32)
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    B, N, dim = P.shape
    M = Q.shape[1]
    ip = np.ascontiguousarray(idx_p, dtype=np.int32)
    iq = np.ascontiguousarray(idx_q, dtype=np.int32)
    g = np.ascontiguousarray(grad, dtype=np.float32).reshape(-1)
    dP = np.zeros((B, N, dim))
    dQ = np.zeros((B, M, dim))
    rc = _load().oracle_chamfer_bwd(_p(P), _p(Q), B, N, M, dim, _p(ip), _p(iq), _p(g), _p(dP), _p(dQ))
    if rc == 3:
        raise ValueError("nearest index outside [-1, set size)")
    if rc:
        raise ValueError(f"oracle_chamfer_bwd failed ({rc})")
    return dP, dQ


def topk(scores, k):
    """The k largest values of every row of scores [R, n] ("Flash-MaxSim"
    Sec. 4 lists a top-K scan among the forward variants; TileMaxSim's
    retrieval pipeline takes the top-k of the scores). Order: descending
    value, the lower index first among equal values (-0.0 equals +0.0).
    Returns (indices [R, k] int32, values [R, k] float64)."""
    s = np.asarray(scores, dtype=np.float64)
    R, n = s.shape
    if not 0 < k <= n:
        raise ValueError("need 0 < k <= n")
    idx = np.empty((R, k), dtype=np.int32)
    for r in range(R):
        order = np.lexsort((np.arange(n), -s[r]))  # primary: -value, then index
        idx[r] = order[:k]
    return idx, np.take_along_axis(s, idx.astype(np.int64), axis=1)


def two_stage_topk(Q8, q_scale, D8, d_scale, Q16, D16, dtype, k1, k, threads=0):
    """Two-stage INT8 -> f16 / bf16 top-k ("Flash-MaxSim" Sec. 4: the
    two-stage INT8 -> FP16 top-K scan among the forward variants):
      1. INT8 x INT8 scores s8 of every (query, document) (fwd_int8);
      2. the k1 best documents of each query by s8 (topk);
      3. those documents rescored from the f16 / bf16 embeddings (fwd_dense);
      4. the k best of the rescored candidates (topk).
    Q8 / D8 int8 [Nq,Lq,dim] / [Nd,Ld,dim] with per-token scales; Q16 / D16 the
    same shapes as uint16 bits of dtype. Returns (top_idx [Nq,k] int32 document
    indices, top_scores [Nq,k], s8 [Nq,Nd], candidates [Nq,k1], s16 [Nq,k1])."""
    Nq = Q8.shape[0]
    s8, _, _, _ = fwd_int8(Q8, q_scale, D8, d_scale, threads=threads)
    cand, _ = topk(s8, k1)
    s16 = np.empty((Nq, k1), dtype=np.float64)
    for i in range(Nq):
        si, _, _ = fwd_dense(Q16[i:i + 1], D16, dtype, docs=cand[i].astype(np.int64), threads=threads)
        s16[i] = si[0]
    pos, top_scores = topk(s16, k)
    top_idx = np.take_along_axis(cand, pos.astype(np.int64), axis=1)
    return top_idx, top_scores, s8, cand, s16
