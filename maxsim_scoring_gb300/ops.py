"""PyTorch-facing binding of the MaxSim C ABI: argument marshalling only.

Every function here checks shapes / dtypes, allocates outputs and workspace
with torch on the tensors' device, and calls the entry point of the same name
in libmaxsim.so on the current CUDA stream. All arithmetic happens in the
CUDA kernels behind that call.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _native

_DT = {torch.float16: _native.F16, torch.bfloat16: _native.BF16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _contig(t: Optional[torch.Tensor], name: str, dtype=None, device=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t.contiguous()


def _mask(m: Optional[torch.Tensor], name: str, device):
    if m is None:
        return None
    if m.dtype == torch.bool:
        m = m.to(torch.uint8)
    return _contig(m, name, torch.uint8, device)


def workspace_size(op: int, Nq: int, Lq: int, Nd: int, Ld: int, dim: int) -> int:
    n = _native.lib().maxsim_workspace_size(op, Nq, Lq, Nd, Ld, dim)
    if n == ctypes_size_max():
        raise ValueError("invalid shape for maxsim_workspace_size")
    return int(n)


def ctypes_size_max() -> int:
    import ctypes
    return ctypes.c_size_t(-1).value


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]):
    if nbytes == 0:
        return None, 0
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        return ws, ws.numel() * ws.element_size()
    t = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return t, nbytes


def maxsim_fwd(Q: torch.Tensor, D: torch.Tensor, q_mask=None, d_mask=None, *, want_argmax: bool = False,
               scores: Optional[torch.Tensor] = None, argmax: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None):
    """scores [Nq, Nd] (and argmax [Nq*Nd, Lq] int32) for Q [Nq,Lq,d], D [Nd,Ld,d]."""
    if Q.dtype not in _DT or D.dtype != Q.dtype:
        raise TypeError("Q and D must both be float16 or both bfloat16")
    dev = Q.device
    Q, D = _contig(Q, "Q"), _contig(D, "D", device=dev)
    Nq, Lq, dim = Q.shape
    Nd, Ld, dim2 = D.shape
    if dim2 != dim:
        raise ValueError("Q and D embedding dimensions differ")
    qm, dm = _mask(q_mask, "q_mask", dev), _mask(d_mask, "d_mask", dev)
    if scores is None:
        scores = torch.empty((Nq, Nd), dtype=torch.float32, device=dev)
    if want_argmax and argmax is None:
        argmax = torch.empty((Nq * Nd, Lq), dtype=torch.int32, device=dev)
    ws, nbytes = _workspace(workspace_size(_native.OP_FWD, Nq, Lq, Nd, Ld, dim), dev, workspace)
    rc = _native.lib().maxsim_fwd(_ptr(Q), _ptr(D), _DT[Q.dtype], Nq, Lq, Nd, Ld, dim, _ptr(qm), _ptr(dm),
                                  _ptr(scores), _ptr(argmax), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_fwd")
    return scores, argmax


def maxsim_fwd_varlen(Q: torch.Tensor, cu_seqlens_q: Optional[torch.Tensor], max_lq: int, D: torch.Tensor,
                      cu_seqlens_d: torch.Tensor, q_mask=None, d_mask=None, *, want_argmax: bool = False,
                      scores: Optional[torch.Tensor] = None, argmax: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None):
    """Packed documents D [total_d, d] with cu_seqlens_d [Nd+1] (int32).

    Q is dense [Nq, max_lq, d] when cu_seqlens_q is None, else packed
    [total_q, d]. Returns scores [Nq, Nd] (and argmax [Nq*Nd, max_lq]).
    """
    if Q.dtype not in _DT or D.dtype != Q.dtype:
        raise TypeError("Q and D must both be float16 or both bfloat16")
    dev = Q.device
    Q, D = _contig(Q, "Q"), _contig(D, "D", device=dev)
    cu_d = _contig(cu_seqlens_d, "cu_seqlens_d", torch.int32, dev)
    cu_q = _contig(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev)
    dim = Q.shape[-1]
    if D.dim() != 2 or D.shape[1] != dim:
        raise ValueError("D must be packed [total_d, dim]")
    Nd = cu_d.numel() - 1
    Nq = (cu_q.numel() - 1) if cu_q is not None else Q.shape[0]
    if cu_q is None and (Q.dim() != 3 or Q.shape[1] != max_lq):
        raise ValueError("dense Q must be [Nq, max_lq, dim]")
    total_d = D.shape[0]
    qm, dm = _mask(q_mask, "q_mask", dev), _mask(d_mask, "d_mask", dev)
    if scores is None:
        scores = torch.empty((Nq, Nd), dtype=torch.float32, device=dev)
    if want_argmax and argmax is None:
        argmax = torch.empty((Nq * Nd, max_lq), dtype=torch.int32, device=dev)
    ws, nbytes = _workspace(workspace_size(_native.OP_FWD_VARLEN, Nq, max_lq, Nd, total_d, dim), dev, workspace)
    rc = _native.lib().maxsim_fwd_varlen(_ptr(Q), _ptr(cu_q), max_lq, _ptr(D), _ptr(cu_d), total_d, _DT[Q.dtype], Nq,
                                         Nd, dim, _ptr(qm), _ptr(dm), _ptr(scores), _ptr(argmax), _ptr(ws), nbytes,
                                         _stream(dev))
    _native.check(rc, "maxsim_fwd_varlen")
    return scores, argmax


def maxsim_score_pairs_packed(Q: torch.Tensor, cu_seqlens_q: Optional[torch.Tensor], max_lq: int, D: torch.Tensor,
                              cu_seqlens_d: torch.Tensor, pairs: torch.Tensor, q_mask=None, d_mask=None, *,
                              want_argmax: bool = False, scores: Optional[torch.Tensor] = None,
                              argmax: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Scores of the (query, document) pairs `pairs` [num_pairs, 2] (int32)
    over the packed batches of maxsim_fwd_varlen. Returns scores [num_pairs]
    (and argmax [num_pairs, max_lq])."""
    if Q.dtype not in _DT or D.dtype != Q.dtype:
        raise TypeError("Q and D must both be float16 or both bfloat16")
    dev = Q.device
    Q, D = _contig(Q, "Q"), _contig(D, "D", device=dev)
    cu_d = _contig(cu_seqlens_d, "cu_seqlens_d", torch.int32, dev)
    cu_q = _contig(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev)
    pr = _contig(pairs, "pairs", torch.int32, dev)
    if pr.dim() != 2 or pr.shape[1] != 2:
        raise ValueError("pairs must be [num_pairs, 2]")
    dim = Q.shape[-1]
    if D.dim() != 2 or D.shape[1] != dim:
        raise ValueError("D must be packed [total_d, dim]")
    Nd = cu_d.numel() - 1
    Nq = (cu_q.numel() - 1) if cu_q is not None else Q.shape[0]
    if cu_q is None and (Q.dim() != 3 or Q.shape[1] != max_lq):
        raise ValueError("dense Q must be [Nq, max_lq, dim]")
    total_d, n = D.shape[0], pr.shape[0]
    qm, dm = _mask(q_mask, "q_mask", dev), _mask(d_mask, "d_mask", dev)
    if scores is None:
        scores = torch.empty((n,), dtype=torch.float32, device=dev)
    if want_argmax and argmax is None:
        argmax = torch.empty((n, max_lq), dtype=torch.int32, device=dev)
    ws, nbytes = _workspace(workspace_size(_native.OP_SCORE_PAIRS, Nq, max_lq, Nd, n, dim), dev, workspace)
    rc = _native.lib().maxsim_score_pairs_packed(_ptr(Q), _ptr(cu_q), max_lq, _ptr(D), _ptr(cu_d), total_d,
                                                 _DT[Q.dtype], Nq, Nd, dim, _ptr(qm), _ptr(dm), _ptr(pr), n,
                                                 _ptr(scores), _ptr(argmax), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_score_pairs_packed")
    return scores, argmax


def maxsim_bwd(Q: torch.Tensor, D: torch.Tensor, argmax: torch.Tensor, grad_scores: torch.Tensor, q_mask=None, *,
               want_dq: bool = True, want_dd: bool = True, want_csr: bool = False,
               dQ: Optional[torch.Tensor] = None, dD: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None):
    """dQ [Nq,Lq,d] f32, dD [Nd,Ld,d] f32 (and the CSR row_ptr / col)."""
    if Q.dtype not in _DT or D.dtype != Q.dtype:
        raise TypeError("Q and D must both be float16 or both bfloat16")
    dev = Q.device
    Q, D = _contig(Q, "Q"), _contig(D, "D", device=dev)
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    am = _contig(argmax, "argmax", torch.int32, dev)
    g = _contig(grad_scores, "grad_scores", torch.float32, dev)
    if am.numel() != Nq * Nd * Lq or g.numel() != Nq * Nd:
        raise ValueError("argmax must be [Nq*Nd, Lq] and grad_scores [Nq, Nd]")
    qm = _mask(q_mask, "q_mask", dev)
    if dQ is None and want_dq:
        dQ = torch.empty((Nq, Lq, dim), dtype=torch.float32, device=dev)
    if dD is None and want_dd:
        dD = torch.empty((Nd, Ld, dim), dtype=torch.float32, device=dev)
    for t, shape, name in ((dQ, (Nq, Lq, dim), "dQ"), (dD, (Nd, Ld, dim), "dD")):
        if t is not None and (tuple(t.shape) != shape or t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 tensor of shape {shape}")
    row_ptr = torch.empty(Nd * Ld + 1, dtype=torch.int32, device=dev) if want_csr else None
    col = torch.empty(max(1, Nq * Nd * Lq), dtype=torch.int32, device=dev) if want_csr else None
    ws, nbytes = _workspace(workspace_size(_native.OP_BWD, Nq, Lq, Nd, Ld, dim), dev, workspace)
    rc = _native.lib().maxsim_bwd(_ptr(Q), _ptr(D), _DT[Q.dtype], Nq, Lq, Nd, Ld, dim, _ptr(qm), _ptr(am), _ptr(g),
                                  _ptr(dQ), _ptr(dD), _ptr(row_ptr), _ptr(col), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_bwd")
    return dQ, dD, row_ptr, col


def maxsim_bwd_varlen(Q: torch.Tensor, cu_seqlens_q: Optional[torch.Tensor], max_lq: int, D: torch.Tensor,
                      cu_seqlens_d: torch.Tensor, max_ld: int, argmax: torch.Tensor, grad_scores: torch.Tensor,
                      q_mask=None, *, want_dq: bool = True, want_dd: bool = True, want_csr: bool = False,
                      workspace: Optional[torch.Tensor] = None):
    """Gradient of maxsim_fwd_varlen: dQ in Q's layout, dD [total_d, d] (f32),
    and optionally the CSR (row_ptr over D's packed rows, col)."""
    if Q.dtype not in _DT or D.dtype != Q.dtype:
        raise TypeError("Q and D must both be float16 or both bfloat16")
    dev = Q.device
    Q, D = _contig(Q, "Q"), _contig(D, "D", device=dev)
    cu_q = _contig(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev)
    cu_d = _contig(cu_seqlens_d, "cu_seqlens_d", torch.int32, dev)
    dim = Q.shape[-1]
    Nq = (cu_q.numel() - 1) if cu_q is not None else Q.shape[0]
    Nd = cu_d.numel() - 1
    total_d = D.shape[0]
    am = _contig(argmax, "argmax", torch.int32, dev)
    g = _contig(grad_scores, "grad_scores", torch.float32, dev)
    if am.numel() != Nq * Nd * max_lq or g.numel() != Nq * Nd:
        raise ValueError("argmax must be [Nq*Nd, max_lq] and grad_scores [Nq, Nd]")
    qm = _mask(q_mask, "q_mask", dev)
    dQ = torch.empty(Q.shape, dtype=torch.float32, device=dev) if want_dq else None
    dD = torch.empty((total_d, dim), dtype=torch.float32, device=dev) if want_dd else None
    row_ptr = torch.empty(total_d + 1, dtype=torch.int32, device=dev) if want_csr else None
    col = torch.empty(max(1, Nq * Nd * max_lq), dtype=torch.int32, device=dev) if want_csr else None
    ws, nbytes = _workspace(workspace_size(_native.OP_BWD_VARLEN, Nq, max_lq, Nd, total_d, dim), dev, workspace)
    rc = _native.lib().maxsim_bwd_varlen(_ptr(Q), _ptr(cu_q), max_lq, _ptr(D), _ptr(cu_d), total_d, max_ld,
                                         _DT[Q.dtype], Nq, Nd, dim, _ptr(qm), _ptr(am), _ptr(g), _ptr(dQ), _ptr(dD),
                                         _ptr(row_ptr), _ptr(col), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_bwd_varlen")
    return dQ, dD, row_ptr, col


def maxsim_fwd_int8(Q: torch.Tensor, q_scale: torch.Tensor, D: torch.Tensor, d_scale: torch.Tensor, q_mask=None,
                    d_mask=None, *, want_argmax: bool = False, want_win_dot: bool = False,
                    scores: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """INT8 x INT8 scores [Nq, Nd] with per-token float32 scales."""
    dev = Q.device
    Q = _contig(Q, "Q", torch.int8)
    D = _contig(D, "D", torch.int8, dev)
    qs = _contig(q_scale, "q_scale", torch.float32, dev)
    ds = _contig(d_scale, "d_scale", torch.float32, dev)
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D.shape
    qm, dm = _mask(q_mask, "q_mask", dev), _mask(d_mask, "d_mask", dev)
    if scores is None:
        scores = torch.empty((Nq, Nd), dtype=torch.float32, device=dev)
    argmax = torch.empty((Nq * Nd, Lq), dtype=torch.int32, device=dev) if (want_argmax or want_win_dot) else None
    win = torch.empty((Nq * Nd, Lq), dtype=torch.int32, device=dev) if want_win_dot else None
    ws, nbytes = _workspace(workspace_size(_native.OP_FWD_INT8, Nq, Lq, Nd, Ld, dim), dev, workspace)
    rc = _native.lib().maxsim_fwd_int8(_ptr(Q), _ptr(qs), _ptr(D), _ptr(ds), Nq, Lq, Nd, Ld, dim, _ptr(qm), _ptr(dm),
                                       _ptr(scores), _ptr(argmax), _ptr(win), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_fwd_int8")
    return scores, argmax, win


def _points(P: torch.Tensor, Q: torch.Tensor):
    if P.dim() != 3 or Q.dim() != 3 or P.shape[0] != Q.shape[0] or P.shape[2] != Q.shape[2]:
        raise ValueError("P must be [B, N, dim] and Q [B, M, dim]")
    dev = P.device
    return _contig(P, "P", torch.float32), _contig(Q, "Q", torch.float32, dev), dev


def chamfer_fwd(P: torch.Tensor, Q: torch.Tensor, *, workspace: Optional[torch.Tensor] = None):
    """Chamfer distance of B pairs of point sets P [B,N,dim], Q [B,M,dim] (f32).

    Returns (loss [B], dist_p [B,N], idx_p [B,N] i32, dist_q [B,M], idx_q [B,M] i32).
    """
    P, Q, dev = _points(P, Q)
    B, N, dim = P.shape
    M = Q.shape[1]
    loss = torch.empty(B, dtype=torch.float32, device=dev)
    dist_p = torch.empty((B, N), dtype=torch.float32, device=dev)
    idx_p = torch.empty((B, N), dtype=torch.int32, device=dev)
    dist_q = torch.empty((B, M), dtype=torch.float32, device=dev)
    idx_q = torch.empty((B, M), dtype=torch.int32, device=dev)
    ws, nbytes = _workspace(workspace_size(_native.OP_CHAMFER_FWD, B, N, M, 0, dim), dev, workspace)
    rc = _native.lib().maxsim_chamfer_fwd(_ptr(P), _ptr(Q), B, N, M, dim, _ptr(dist_p), _ptr(idx_p), _ptr(dist_q),
                                          _ptr(idx_q), _ptr(loss), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_chamfer_fwd")
    return loss, dist_p, idx_p, dist_q, idx_q


def chamfer_bwd(P: torch.Tensor, Q: torch.Tensor, idx_p: torch.Tensor, idx_q: torch.Tensor, grad_loss: torch.Tensor,
                *, dP: Optional[torch.Tensor] = None, dQ: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None):
    """(dP [B,N,dim], dQ [B,M,dim]) f32 of sum_b grad_loss[b] * CD(P_b, Q_b)."""
    P, Q, dev = _points(P, Q)
    B, N, dim = P.shape
    M = Q.shape[1]
    ip = _contig(idx_p, "idx_p", torch.int32, dev)
    iq = _contig(idx_q, "idx_q", torch.int32, dev)
    g = _contig(grad_loss, "grad_loss", torch.float32, dev)
    if ip.numel() != B * N or iq.numel() != B * M or g.numel() != B:
        raise ValueError("idx_p must be [B, N], idx_q [B, M] and grad_loss [B]")
    if dP is None:
        dP = torch.empty((B, N, dim), dtype=torch.float32, device=dev)
    if dQ is None:
        dQ = torch.empty((B, M, dim), dtype=torch.float32, device=dev)
    for t, shape, name in ((dP, (B, N, dim), "dP"), (dQ, (B, M, dim), "dQ")):
        if tuple(t.shape) != shape or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor of shape {shape}")
    ws, nbytes = _workspace(workspace_size(_native.OP_CHAMFER_BWD, B, N, M, 0, dim), dev, workspace)
    rc = _native.lib().maxsim_chamfer_bwd(_ptr(P), _ptr(Q), B, N, M, dim, _ptr(ip), _ptr(iq), _ptr(g), _ptr(dP),
                                          _ptr(dQ), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_chamfer_bwd")
    return dP, dQ


def maxsim_topk(scores: torch.Tensor, k: int):
    """(values [R, k] f32, indices [R, k] i32): the k largest entries of every
    row of scores [R, n] (f32), descending, the lower index first among ties."""
    s = _contig(scores, "scores", torch.float32)
    if s.dim() != 2:
        raise ValueError("scores must be [rows, n]")
    R, n = s.shape
    idx = torch.empty((R, k), dtype=torch.int32, device=s.device)
    vals = torch.empty((R, k), dtype=torch.float32, device=s.device)
    rc = _native.lib().maxsim_topk(_ptr(s), R, n, k, _ptr(idx), _ptr(vals), _stream(s.device))
    _native.check(rc, "maxsim_topk")
    return vals, idx


def maxsim_two_stage_topk(Q8: torch.Tensor, q_scale: torch.Tensor, D8: torch.Tensor, d_scale: torch.Tensor,
                          Q16: torch.Tensor, D16: torch.Tensor, k1: int, k: int, *, want_stage1: bool = False,
                          workspace: Optional[torch.Tensor] = None):
    """Two-stage INT8 -> f16 / bf16 top-k: (top_idx [Nq,k] i32, top_scores [Nq,k] f32,
    stage1_scores [Nq,Nd] or None, candidates [Nq,k1] or None)."""
    dev = Q8.device
    Q8 = _contig(Q8, "Q8", torch.int8)
    D8 = _contig(D8, "D8", torch.int8, dev)
    qs = _contig(q_scale, "q_scale", torch.float32, dev)
    ds = _contig(d_scale, "d_scale", torch.float32, dev)
    if Q16.dtype not in _DT or D16.dtype != Q16.dtype:
        raise TypeError("Q16 and D16 must both be float16 or both bfloat16")
    Q16, D16 = _contig(Q16, "Q16", device=dev), _contig(D16, "D16", device=dev)
    Nq, Lq, dim = Q8.shape
    Nd, Ld, _ = D8.shape
    if tuple(Q16.shape) != (Nq, Lq, dim) or tuple(D16.shape) != (Nd, Ld, dim):
        raise ValueError("Q16 / D16 must have the shapes of Q8 / D8")
    top_idx = torch.empty((Nq, k), dtype=torch.int32, device=dev)
    top_scores = torch.empty((Nq, k), dtype=torch.float32, device=dev)
    s8 = torch.empty((Nq, Nd), dtype=torch.float32, device=dev) if want_stage1 else None
    cand = torch.empty((Nq, k1), dtype=torch.int32, device=dev) if want_stage1 else None
    ws, nbytes = _workspace(workspace_size(_native.OP_TWO_STAGE, Nq, Lq, Nd, Ld, dim), dev, workspace)
    rc = _native.lib().maxsim_two_stage_topk(_ptr(Q8), _ptr(qs), _ptr(D8), _ptr(ds), _ptr(Q16), _ptr(D16),
                                             _DT[Q16.dtype], Nq, Lq, Nd, Ld, dim, k1, k, _ptr(top_idx),
                                             _ptr(top_scores), _ptr(s8), _ptr(cand), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_two_stage_topk")
    return top_idx, top_scores, s8, cand


def maxsim_fwd_streamed(Q: torch.Tensor, D_host: torch.Tensor, q_mask=None, *, block_docs: int = 20_000,
                        scores: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Scores [Nq, Nd] of a device query batch Q [Nq,Lq,d] against a corpus
    D_host [Nd,Ld,d] in host memory (pin it for copy/compute overlap),
    streamed in blocks of block_docs documents. The copies are asynchronous:
    keep D_host alive and unchanged until the current stream has passed this
    call (synchronise, or wait on an event recorded after it)."""
    if Q.dtype not in _DT or D_host.dtype != Q.dtype:
        raise TypeError("Q and D_host must both be float16 or both bfloat16")
    if D_host.is_cuda or not D_host.is_contiguous():
        raise ValueError("D_host must be a contiguous host tensor")
    dev = Q.device
    Q = _contig(Q, "Q")
    Nq, Lq, dim = Q.shape
    Nd, Ld, _ = D_host.shape
    qm = _mask(q_mask, "q_mask", dev)
    if scores is None:
        scores = torch.empty((Nq, Nd), dtype=torch.float32, device=dev)
    ws, nbytes = _workspace(workspace_size(_native.OP_FWD_STREAMED, Nq, Lq, min(block_docs, max(Nd, 1)), Ld, dim),
                            dev, workspace)
    rc = _native.lib().maxsim_fwd_streamed(_ptr(Q), D_host.data_ptr(), _DT[Q.dtype], Nq, Lq, Nd, Ld, dim, block_docs,
                                           _ptr(qm), _ptr(scores), _ptr(ws), nbytes, _stream(dev))
    _native.check(rc, "maxsim_fwd_streamed")
    return scores


def maxsim_fwd_varlen_streamed(Q: torch.Tensor, cu_seqlens_q: Optional[torch.Tensor], max_lq: int,
                               D_host: torch.Tensor, cu_seqlens_d_host: torch.Tensor, q_mask=None, *,
                               block_docs: int = 20_000, block_tokens: int = 1 << 22,
                               scores: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Scores [Nq, Nd] of device queries against a packed corpus in host
    memory: D_host [total_d, d] rows and cu_seqlens_d_host [Nd+1] (int32, host),
    streamed in blocks of whole documents. Keep the host tensors alive and
    unchanged until the current stream has passed this call."""
    if Q.dtype not in _DT or D_host.dtype != Q.dtype:
        raise TypeError("Q and D_host must both be float16 or both bfloat16")
    if D_host.is_cuda or cu_seqlens_d_host.is_cuda or not D_host.is_contiguous():
        raise ValueError("D_host and cu_seqlens_d_host must be contiguous host tensors")
    if cu_seqlens_d_host.dtype != torch.int32 or not cu_seqlens_d_host.is_contiguous():
        raise TypeError("cu_seqlens_d_host must be a contiguous int32 host tensor")
    dev = Q.device
    Q = _contig(Q, "Q")
    cu_q = _contig(cu_seqlens_q, "cu_seqlens_q", torch.int32, dev)
    dim = Q.shape[-1]
    Nq = (cu_q.numel() - 1) if cu_q is not None else Q.shape[0]
    Nd = cu_seqlens_d_host.numel() - 1
    total_d = D_host.shape[0]
    qm = _mask(q_mask, "q_mask", dev)
    if scores is None:
        scores = torch.empty((Nq, Nd), dtype=torch.float32, device=dev)
    bd = min(block_docs, max(Nd, 1))
    ws, nbytes = _workspace(workspace_size(_native.OP_FWD_VARLEN_STREAMED, Nq, max_lq, bd, block_tokens, dim), dev,
                            workspace)
    rc = _native.lib().maxsim_fwd_varlen_streamed(_ptr(Q), _ptr(cu_q), max_lq, D_host.data_ptr(),
                                                  cu_seqlens_d_host.data_ptr(), total_d, _DT[Q.dtype], Nq, Nd, dim,
                                                  _ptr(qm), block_docs, block_tokens, _ptr(scores), _ptr(ws), nbytes,
                                                  _stream(dev))
    _native.check(rc, "maxsim_fwd_varlen_streamed")
    return scores


def device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device status word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return int(_native.lib().maxsim_device_status(_stream(dev)))


def debug_inject_wait_timeout(limit_ns: int) -> None:
    """Fault-handling test hook: the next forward launch from this process
    waits, in its epilogue, on a barrier nothing arrives at and gives up after
    limit_ns, recording MAXSIM_ERR_TIMEOUT (read it with device_status())."""
    _native.check(_native.lib().maxsim_debug_inject_wait_timeout(int(limit_ns)), "maxsim_debug_inject_wait_timeout")
