"""The packed-layout backward (maxsim_bwd_varlen) against the oracle's
backward, which is applied to the same data laid out densely (documents and
queries padded; padded rows are never selected, so they carry no gradient),
and against the dense backward where both layouts coincide."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from maxsim_scoring_gb300 import maxsim_varlen, ops
from tests.gpu_util import assert_grad, dev, dev_bits

pytestmark = pytest.mark.gpu


def packed(seed, lens, dim, dtype, tid):
    cu = np.zeros(len(lens) + 1, np.int64)
    np.cumsum(lens, out=cu[1:])
    return datagen.gaussian_rows(seed, tid, int(cu[-1]), dim, dtype), cu


def to_dense(rows, cu, width, dim):
    out = np.zeros((len(cu) - 1, width, dim), dtype=rows.dtype)
    for i in range(len(cu) - 1):
        out[i, :cu[i + 1] - cu[i]] = rows[cu[i]:cu[i + 1]]
    return out


def oracle_bwd_packed(Q, cu_q, max_lq, D, cu_d, max_ld, dtype, argmax, g, q_mask=None):
    dim = D.shape[-1]
    Qd = to_dense(Q, cu_q, max_lq, dim) if cu_q is not None else Q
    Dd = to_dense(D, cu_d, max_ld, dim)
    qm = None
    if q_mask is not None:
        qm = to_dense(q_mask.reshape(-1, 1), cu_q, max_lq, 1)[..., 0] if cu_q is not None else q_mask
    dQd, dDd, rp, col = oracle.bwd(Qd, Dd, dtype, argmax, g, q_mask=qm)
    Nd = len(cu_d) - 1
    dD = np.concatenate([dDd[j, :cu_d[j + 1] - cu_d[j]] for j in range(Nd)]) if cu_d[-1] else np.zeros((0, dim))
    rows = np.concatenate([j * max_ld + np.arange(cu_d[j + 1] - cu_d[j]) for j in range(Nd)] + [[Nd * max_ld]])
    dQ = np.concatenate([dQd[i, :cu_q[i + 1] - cu_q[i]] for i in range(len(cu_q) - 1)]) if cu_q is not None else dQd
    return dQ, dD, rp[rows.astype(np.int64)], col


def run(Qt, cu_q, max_lq, Dt, cu_d, max_ld, g, q_mask=None):
    s, am = ops.maxsim_fwd_varlen(Qt, None if cu_q is None else dev(cu_q.astype(np.int32)), max_lq, Dt,
                                  dev(cu_d.astype(np.int32)), q_mask, want_argmax=True)
    dQ, dD, rp, col = ops.maxsim_bwd_varlen(Qt, None if cu_q is None else dev(cu_q.astype(np.int32)), max_lq, Dt,
                                            dev(cu_d.astype(np.int32)), max_ld, am, dev(g), q_mask, want_csr=True)
    assert ops.device_status() == 0
    return am.cpu().numpy(), dQ, dD, rp.cpu().numpy(), col.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_packed_documents_dense_queries(dtype):
    rng = np.random.default_rng(91)
    Nq, Lq, dim = 5, 40, 128
    dlens = rng.integers(0, 301, size=23)
    dlens[4] = 0
    Q = datagen.gaussian_rows(91, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D, cu_d = packed(91, dlens, dim, dtype, 2)
    g = rng.standard_normal((Nq, len(dlens))).astype(np.float32)
    max_ld = int(dlens.max())
    am, dQ, dD, rp, col = run(dev_bits(Q, dtype), None, Lq, dev_bits(D, dtype), cu_d, max_ld, g)
    rdQ, rdD, rrp, rcol = oracle_bwd_packed(Q, None, Lq, D, cu_d, max_ld, dtype, am, g)
    assert np.array_equal(rp, rrp) and np.array_equal(col[:rrp[-1]], rcol)
    assert_grad(dQ, rdQ)
    assert_grad(dD, rdD)


def test_packed_queries_with_mask():
    rng = np.random.default_rng(93)
    dtype, dim = "bf16", 64
    qlens = np.array([7, 0, 32, 19, 64])
    dlens = rng.integers(1, 200, size=17)
    Q, cu_q = packed(93, qlens, dim, dtype, 1)
    D, cu_d = packed(93, dlens, dim, dtype, 2)
    qm = (rng.random(int(cu_q[-1])) > 0.25).astype(np.uint8)
    g = rng.standard_normal((len(qlens), len(dlens))).astype(np.float32)
    max_lq, max_ld = int(qlens.max()), int(dlens.max())
    am, dQ, dD, rp, col = run(dev_bits(Q, dtype), cu_q, max_lq, dev_bits(D, dtype), cu_d, max_ld, g, dev(qm))
    rdQ, rdD, rrp, rcol = oracle_bwd_packed(Q, cu_q, max_lq, D, cu_d, max_ld, dtype, am, g, q_mask=qm)
    assert np.array_equal(rp, rrp) and np.array_equal(col[:rrp[-1]], rcol)
    assert tuple(dQ.shape) == (int(cu_q[-1]), dim)
    assert_grad(dQ, rdQ)
    assert_grad(dD, rdD)


def test_uniform_lengths_equal_the_dense_backward():
    dtype, dim, Nq, Lq, Nd, Ld = "f16", 128, 4, 32, 12, 96
    rng = np.random.default_rng(97)
    Q = datagen.gaussian_rows(97, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(97, 2, Nd * Ld, dim, dtype).reshape(Nd, Ld, dim)
    g = rng.standard_normal((Nq, Nd)).astype(np.float32)
    Qt, Dt = dev_bits(Q, dtype), dev_bits(D, dtype)
    _, am = ops.maxsim_fwd(Qt, Dt, want_argmax=True)
    dQ, dD, rp, col = ops.maxsim_bwd(Qt, Dt, am, dev(g), want_csr=True)
    cu = dev((np.arange(Nd + 1) * Ld).astype(np.int32))
    vQ, vD, vrp, vcol = ops.maxsim_bwd_varlen(Qt, None, Lq, Dt.reshape(Nd * Ld, dim), cu, Ld, am, dev(g),
                                              want_csr=True)
    assert ops.device_status() == 0
    assert torch.equal(dQ, vQ) and torch.equal(dD.reshape(Nd * Ld, dim), vD)
    assert torch.equal(rp, vrp) and torch.equal(col, vcol)


def test_autograd_varlen():
    dtype, dim = "bf16", 128
    rng = np.random.default_rng(101)
    Nq, Lq = 3, 32
    dlens = rng.integers(1, 150, size=9)
    Q = datagen.gaussian_rows(101, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D, cu_d = packed(101, dlens, dim, dtype, 2)
    Qt = dev_bits(Q, dtype).requires_grad_(True)
    Dt = dev_bits(D, dtype).requires_grad_(True)
    cu = dev(cu_d.astype(np.int32))
    w = torch.randn(Nq, len(dlens), device="cuda")
    (maxsim_varlen(Qt, None, Lq, Dt, cu, int(dlens.max())) * w).sum().backward()
    _, am = ops.maxsim_fwd_varlen(Qt.detach(), None, Lq, Dt.detach(), cu, want_argmax=True)
    dQ, dD, _, _ = ops.maxsim_bwd_varlen(Qt.detach(), None, Lq, Dt.detach(), cu, int(dlens.max()), am, w)
    assert torch.equal(Qt.grad, dQ.to(Qt.dtype)) and torch.equal(Dt.grad, dD.to(Dt.dtype))


def test_bad_argmax_is_reported_and_skipped():
    dtype, dim = "f16", 64
    rng = np.random.default_rng(103)
    dlens = np.array([10, 5, 20])
    Q = datagen.gaussian_rows(103, 1, 2 * 8, dim, dtype).reshape(2, 8, dim)
    D, cu_d = packed(103, dlens, dim, dtype, 2)
    Qt, Dt, cu = dev_bits(Q, dtype), dev_bits(D, dtype), dev(cu_d.astype(np.int32))
    _, am = ops.maxsim_fwd_varlen(Qt, None, 8, Dt, cu, want_argmax=True)
    bad = am.clone()
    bad[1, 3] = 7  # document 1 has 5 rows
    g = dev(rng.standard_normal((2, 3)).astype(np.float32))
    dQ, dD, _, _ = ops.maxsim_bwd_varlen(Qt, None, 8, Dt, cu, 20, bad, g)
    assert ops.device_status() == 6
    skip = am.clone()
    skip[1, 3] = -1
    rQ, rD, _, _ = ops.maxsim_bwd_varlen(Qt, None, 8, Dt, cu, 20, skip, g)
    assert ops.device_status() == 0
    assert torch.equal(dD, rD)
