"""Failure detection without a GPU fault: a device-side bounded wait that runs
out is reported through the status word, the kernel returns, and the next
call is correct.

The forward's epilogue is made to wait on an mbarrier that nothing arrives at
(maxsim_debug_inject_wait_timeout); no other wait is shortened, so the copies
and MMAs the other roles already issued land before the CTAs leave. Nothing
traps and no wait is endless."""
import time

import numpy as np
import pytest
import torch

import datagen
import oracle
from maxsim_scoring_gb300 import _native, ops
from tests.gpu_util import assert_argmax, assert_scores, dev, dev_bits

pytestmark = pytest.mark.gpu


def _varlen_problem(seed=61, Nq=4, Lq=32, lens=(40, 0, 300, 128, 17, 256, 33), dim=128):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Q = datagen.gaussian_rows(seed, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(seed, 2, int(cu[-1]), dim, "f16")
    return Q, D, cu


def test_hook_rejects_bad_limits():
    for bad in (0, 2_000_000_001):
        assert _native.lib().maxsim_debug_inject_wait_timeout(bad) == 1  # MAXSIM_ERR_INVALID_ARG


@pytest.mark.parametrize("want_argmax", [False, True])
def test_forward_wait_timeout_reported_then_next_call_correct(want_argmax):
    Qb, Db, cu = _varlen_problem()
    Nq, Lq = Qb.shape[:2]
    Q, D, cud = dev_bits(Qb, "f16"), dev_bits(Db, "f16"), dev(cu)
    assert ops.device_status() == 0
    ops.debug_inject_wait_timeout(1_000_000)  # 1 ms
    t0 = time.perf_counter()
    ops.maxsim_fwd_varlen(Q, None, Lq, D, cud, want_argmax=want_argmax)
    st = ops.device_status()  # synchronises: the kernel has returned
    elapsed = time.perf_counter() - t0
    assert st == 4, _native.STATUS.get(st, st)  # MAXSIM_ERR_TIMEOUT
    assert ops.device_status() == 0  # read and cleared
    assert elapsed < 1.5, f"the aborted launch took {elapsed:.3f} s (the normal wait limit is 2 s)"
    # the hook is one-shot: the next call runs normally and is correct
    s, a = ops.maxsim_fwd_varlen(Q, None, Lq, D, cud, want_argmax=True)
    assert ops.device_status() == 0
    ref_s, ref_a, gap = oracle.fwd_packed(Qb.reshape(-1, Qb.shape[2]), np.arange(Nq + 1, dtype=np.int64) * Lq, Db,
                                          cu.astype(np.int64), "f16")
    assert_scores(s, ref_s, Lq)
    assert_argmax(a, ref_a, gap)
    torch.cuda.synchronize()


def test_int8_pair_forward_wait_timeout_reported():
    # the two-CTA (cluster) forward takes the same abort path on both CTAs
    Nq, Lq, Nd, Ld, dim = 1, 1024, 6, 200, 128
    q, qs = datagen.int8_rows(62, 1, Nq * Lq, dim)
    d, ds = datagen.int8_rows(62, 2, Nd * Ld, dim)
    Q8, D8 = q.reshape(Nq, Lq, dim), d.reshape(Nd, Ld, dim)
    args = (dev(Q8), dev(qs.reshape(Nq, Lq)), dev(D8), dev(ds.reshape(Nd, Ld)))
    ops.debug_inject_wait_timeout(1_000_000)
    ops.maxsim_fwd_int8(*args)
    assert ops.device_status() == 4
    s, _, _ = ops.maxsim_fwd_int8(*args)
    assert ops.device_status() == 0
    ref_s, _, _, _ = oracle.fwd_int8(Q8, qs.reshape(Nq, Lq), D8, ds.reshape(Nd, Ld))
    assert_scores(s, ref_s, Lq)
