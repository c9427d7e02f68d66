"""Fused MaxSim (ColBERT / ColPali late interaction) for GB300.

    score[i, j] = sum_s max_t <Q[i, s], D[j, t]>

The compute lives in libmaxsim.so (hand-written sm_103a kernels behind the C
ABI of include/maxsim.h); this package is its PyTorch-facing binding plus an
autograd wrapper.
"""
from .ops import (chamfer_bwd, chamfer_fwd, device_status, maxsim_bwd, maxsim_bwd_varlen,  # noqa: F401
                  maxsim_fwd, maxsim_fwd_int8, maxsim_fwd_streamed, maxsim_fwd_varlen, maxsim_fwd_varlen_streamed,
                  maxsim_score_pairs_packed,
                  maxsim_topk, maxsim_two_stage_topk, workspace_size)
from .autograd import chamfer_distance, maxsim, maxsim_varlen  # noqa: F401

__all__ = ["maxsim", "maxsim_varlen", "maxsim_fwd", "maxsim_fwd_varlen", "maxsim_score_pairs_packed", "maxsim_bwd",
           "maxsim_bwd_varlen", "maxsim_fwd_int8", "maxsim_fwd_streamed", "maxsim_fwd_varlen_streamed", "maxsim_topk", "maxsim_two_stage_topk",
           "chamfer_fwd", "chamfer_bwd", "chamfer_distance", "workspace_size", "device_status"]
