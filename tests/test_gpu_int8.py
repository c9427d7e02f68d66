"""Parity of the INT8 x INT8 forward (maxsim_fwd_int8) with the CPU oracle."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from maxsim_scoring_gb300 import ops
from tests.gpu_util import assert_argmax, assert_scores, dev

pytestmark = pytest.mark.gpu


def run_int8(Q, qs, D, ds, q_mask=None, d_mask=None, exact=False, exact_scores=True):
    Nq, Lq, dim = Q.shape
    s, a, w = ops.maxsim_fwd_int8(dev(Q), dev(qs), dev(D), dev(ds), dev(q_mask), dev(d_mask), want_win_dot=True)
    s_only, _, _ = ops.maxsim_fwd_int8(dev(Q), dev(qs), dev(D), dev(ds), dev(q_mask), dev(d_mask))
    assert ops.device_status() == 0
    ref_s, ref_a, ref_w, gap = oracle.fwd_int8(Q, qs, D, ds, q_mask=q_mask, d_mask=d_mask)
    if exact:
        if exact_scores:
            assert np.array_equal(s.cpu().numpy().astype(np.float64), ref_s)
        else:
            assert_scores(s, ref_s, Lq)
        assert np.array_equal(a.cpu().numpy(), ref_a)
    else:
        assert_scores(s, ref_s, Lq)
        assert_argmax(a, ref_a, gap)
    got_a = a.cpu().numpy()
    same = got_a == ref_a
    assert np.array_equal(w.cpu().numpy()[same], ref_w[same])  # exact int32 dot at the argmax
    assert torch.equal(s, s_only)
    return s, a, w


@pytest.mark.parametrize("shape", [(2, 32, 5, 300, 128), (3, 8, 4, 130, 32), (1, 64, 3, 257, 256),
                                   (2, 40, 3, 100, 96),
                                   # two or more row blocks: the two-CTA (cta_group::2) path, where each
                                   # CTA holds half of every document tile; 1280 rows leave the last
                                   # pair half empty
                                   (40, 32, 3, 140, 128), (1, 1024, 3, 200, 128)])
def test_int8_integer_exact(shape):
    # unit / power-of-two scales and |dot| * Lq < 2^24: every similarity and
    # every partial sum is exact in fp32, so scores, argmax (ties included)
    # and win_dot must match bit for bit
    Nq, Lq, Nd, Ld, dim = shape
    rng = np.random.default_rng(sum(shape))
    Q = rng.integers(-127, 128, size=(Nq, Lq, dim)).astype(np.int8)
    D = rng.integers(-7, 8, size=(Nd, Ld, dim)).astype(np.int8)
    qs = np.ones((Nq, Lq), np.float32)
    ds = np.where(rng.random((Nd, Ld)) > 0.5, 1.0, 0.5).astype(np.float32)  # powers of two stay exact
    qm = (rng.random((Nq, Lq)) > 0.2).astype(np.uint8)
    dm = (rng.random((Nd, Ld)) > 0.2).astype(np.uint8)
    # scores are sums of Lq such values: exact in fp32 only while they stay
    # well inside the 24-bit significand (half-integers need one bit more)
    exact_scores = Lq * 127 * 7 * dim < (1 << 22)
    run_int8(Q, qs, D, ds, exact=True, exact_scores=exact_scores)
    run_int8(Q, qs, D, ds, q_mask=qm, d_mask=dm, exact=True, exact_scores=exact_scores)


def test_int8_extreme_values_accumulate_exactly():
    # all entries +-127 at dim 256: |dot| up to 127^2 * 256 = 4,129,024 < 2^24
    Nq, Lq, Nd, Ld, dim = 1, 32, 3, 64, 256
    rng = np.random.default_rng(1)
    Q = np.where(rng.random((Nq, Lq, dim)) > 0.5, 127, -127).astype(np.int8)
    D = np.where(rng.random((Nd, Ld, dim)) > 0.5, 127, -127).astype(np.int8)
    D[0, 5] = Q[0, 0]  # the largest possible dot appears
    qs, ds = np.ones((Nq, Lq), np.float32), np.ones((Nd, Ld), np.float32)
    _, a, w = run_int8(Q, qs, D, ds, exact=True, exact_scores=False)  # sums of 32 such dots exceed 2^24
    assert int(w.cpu().numpy()[0, 0]) == 127 * 127 * 256


@pytest.mark.parametrize("Lq", [32, 1024])
def test_int8_quantised_gaussian(Lq):
    Nq, Nd, Ld, dim = 2, 6, 333, 128
    q, qs = datagen.int8_rows(7, 1, Nq * Lq, dim)
    d, ds = datagen.int8_rows(7, 2, Nd * Ld, dim)
    Q, D = q.reshape(Nq, Lq, dim), d.reshape(Nd, Ld, dim)
    qm = datagen.mask_drop_tail(7, 4, Nq, Lq, Lq // 4)
    dm = datagen.mask_random_subset(7, 5, Nd, Ld, 60)
    run_int8(Q, qs.reshape(Nq, Lq), D, ds.reshape(Nd, Ld))
    run_int8(Q, qs.reshape(Nq, Lq), D, ds.reshape(Nd, Ld), q_mask=qm, d_mask=dm)


def test_int8_win_dot_needs_argmax():
    from maxsim_scoring_gb300 import _native
    Q = torch.zeros((1, 4, 32), dtype=torch.int8, device="cuda")
    qs = torch.ones((1, 4), device="cuda")
    D = torch.zeros((2, 5, 32), dtype=torch.int8, device="cuda")
    ds = torch.ones((2, 5), device="cuda")
    sc = torch.empty((1, 2), device="cuda")
    win = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    rc = _native.lib().maxsim_fwd_int8(Q.data_ptr(), qs.data_ptr(), D.data_ptr(), ds.data_ptr(), 1, 4, 2, 5, 32,
                                       None, None, sc.data_ptr(), None, win.data_ptr(), None, 0,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 1
