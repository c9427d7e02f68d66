"""torch.autograd integration: the forward saves the argmax, the backward runs
the inverse-argmax CSR kernels ("Flash-MaxSim" Sec. 4.2: built at runtime from
the saved argmax, inside autograd)."""
from __future__ import annotations

import torch

from . import ops


class _MaxSim(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, D, q_mask, d_mask):
        scores, argmax = ops.maxsim_fwd(Q, D, q_mask, d_mask, want_argmax=True)
        ctx.save_for_backward(Q, D, argmax, q_mask if q_mask is not None else torch.empty(0))
        ctx.has_qmask = q_mask is not None
        return scores

    @staticmethod
    def backward(ctx, grad_scores):
        Q, D, argmax, q_mask = ctx.saved_tensors
        need_q, need_d = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        dQ, dD, _, _ = ops.maxsim_bwd(Q, D, argmax, grad_scores.float().contiguous(),
                                      q_mask if ctx.has_qmask else None, want_dq=need_q, want_dd=need_d)
        dQ = dQ.to(Q.dtype) if dQ is not None else None
        dD = dD.to(D.dtype) if dD is not None else None
        return dQ, dD, None, None


def maxsim(Q: torch.Tensor, D: torch.Tensor, q_mask=None, d_mask=None) -> torch.Tensor:
    """Differentiable MaxSim scores [Nq, Nd] for Q [Nq,Lq,d], D [Nd,Ld,d]."""
    return _MaxSim.apply(Q, D, q_mask, d_mask)


class _Chamfer(torch.autograd.Function):
    @staticmethod
    def forward(ctx, P, Q):
        loss, _, idx_p, _, idx_q = ops.chamfer_fwd(P, Q)
        ctx.save_for_backward(P, Q, idx_p, idx_q)
        return loss

    @staticmethod
    def backward(ctx, grad_loss):
        P, Q, idx_p, idx_q = ctx.saved_tensors
        dP, dQ = ops.chamfer_bwd(P, Q, idx_p, idx_q, grad_loss.float().contiguous())
        return dP, dQ


def chamfer_distance(P: torch.Tensor, Q: torch.Tensor) -> torch.Tensor:
    """Differentiable Chamfer distance [B] of point sets P [B,N,dim], Q [B,M,dim]
    (float32): the forward saves the nearest indices, the backward routes the
    gradient through their inverse ("Flash-MaxSim" Sec. 4.2.4)."""
    return _Chamfer.apply(P, Q)


class _MaxSimVarlen(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, cu_seqlens_q, max_lq, D, cu_seqlens_d, max_ld):
        scores, argmax = ops.maxsim_fwd_varlen(Q, cu_seqlens_q, max_lq, D, cu_seqlens_d, want_argmax=True)
        ctx.save_for_backward(Q, D, argmax, cu_seqlens_d,
                              cu_seqlens_q if cu_seqlens_q is not None else torch.empty(0, dtype=torch.int32))
        ctx.has_cu_q = cu_seqlens_q is not None
        ctx.max_lq, ctx.max_ld = max_lq, max_ld
        return scores

    @staticmethod
    def backward(ctx, grad_scores):
        Q, D, argmax, cu_d, cu_q = ctx.saved_tensors
        dQ, dD, _, _ = ops.maxsim_bwd_varlen(Q, cu_q if ctx.has_cu_q else None, ctx.max_lq, D, cu_d, ctx.max_ld, argmax,
                                             grad_scores.float().contiguous(), want_dq=ctx.needs_input_grad[0],
                                             want_dd=ctx.needs_input_grad[3])
        dQ = dQ.to(Q.dtype) if dQ is not None else None
        dD = dD.to(D.dtype) if dD is not None else None
        return dQ, None, None, dD, None, None


def maxsim_varlen(Q: torch.Tensor, cu_seqlens_q, max_lq: int, D: torch.Tensor, cu_seqlens_d: torch.Tensor,
                  max_ld: int) -> torch.Tensor:
    """Differentiable MaxSim over packed documents (and optionally packed
    queries): scores [Nq, Nd]."""
    return _MaxSimVarlen.apply(Q, cu_seqlens_q, max_lq, D, cu_seqlens_d, max_ld)
