"""Fused MaxSim (ColBERT / ColPali late interaction) for GB300.

    score[i, j] = sum_s max_t <Q[i, s], D[j, t]>

The compute lives in libmaxsim.so (hand-written sm_103a kernels behind the C
ABI of include/maxsim.h); this package is its PyTorch-facing binding plus an
autograd wrapper.
"""
from .ops import (device_status, maxsim_bwd, maxsim_fwd, maxsim_fwd_int8, maxsim_fwd_varlen,  # noqa: F401
                  maxsim_score_pairs_packed, workspace_size)
from .autograd import maxsim  # noqa: F401

__all__ = ["maxsim", "maxsim_fwd", "maxsim_fwd_varlen", "maxsim_score_pairs_packed", "maxsim_bwd", "maxsim_fwd_int8",
           "workspace_size", "device_status"]
