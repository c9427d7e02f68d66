"""maxsim_fwd_varlen_noalloc: the forward for callers that cannot allocate
device memory (no workspace argument; its scratch is a fixed array inside the
library). Called through the C ABI and compared with maxsim_fwd_varlen, which
takes a caller-allocated workspace. This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import datagen
from maxsim_scoring_gb300 import _native, ops
from tests.gpu_util import dev, dev_bits

pytestmark = pytest.mark.gpu


def _inputs(seed, lens, Nq, Lq, dim):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Q = datagen.gaussian_rows(seed, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(seed, 2, int(cu[-1]), dim, "f16")
    return dev_bits(Q, "f16"), dev_bits(D, "f16"), dev(cu)


def _noalloc(Q, cu_q, max_lq, D, cu_d, Nq, q_mask=None, want_argmax=True):
    Nd = cu_d.numel() - 1
    dim = D.shape[1]
    scores = torch.empty((Nq, Nd), dtype=torch.float32, device=D.device)
    argmax = torch.empty((Nq * Nd, max_lq), dtype=torch.int32, device=D.device) if want_argmax else None
    rc = _native.lib().maxsim_fwd_varlen_noalloc(
        Q.data_ptr(), None if cu_q is None else cu_q.data_ptr(), max_lq, D.data_ptr(), cu_d.data_ptr(), D.shape[0],
        _native.F16, Nq, Nd, dim, None if q_mask is None else q_mask.data_ptr(), None, scores.data_ptr(),
        None if argmax is None else argmax.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc, scores, argmax


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [
        (3, np.array([40, 0, 300, 128, 1, 77, 256]), 4, 40, 128),   # padded query rows
        (4, np.array([32, 33, 290, 0, 5]), 3, 32, 64),               # different shape, same scratch
    ]
    for seed, lens, Nq, Lq, dim in cases:  # two calls in a row on the shared scratch
        Q, D, cu = _inputs(seed, lens, Nq, Lq, dim)
        rc, s_na, a_na = _noalloc(Q, None, Lq, D, cu, Nq)
        assert rc == 0, _native.STATUS.get(rc, rc)
        s_ws, a_ws = ops.maxsim_fwd_varlen(Q, None, Lq, D, cu, want_argmax=True)
        assert ops.device_status() == 0
        assert torch.equal(s_na, s_ws)  # same plan, same kernel, same inputs: identical bits
        assert torch.equal(a_na, a_ws)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    Q, D, cu = _inputs(5, np.array([10, 20]), 1, 8, 128)
    # 70,000 queries of 32 rows need far more than the fixed scratch: rejected before any launch
    rc, _, _ = _noalloc(Q, None, 32, D, cu, 70_000, want_argmax=False)
    assert rc == 2
    assert ops.device_status() == 0
