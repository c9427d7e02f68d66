"""Parity of the packed forward (maxsim_fwd_varlen) and of the backward
(maxsim_bwd) with the CPU oracle."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from maxsim_scoring_gb300 import ops
from tests.gpu_util import (assert_argmax, assert_grad, assert_grad_rounded, assert_scores, dev, dev_bits,
                            integer_rows)

pytestmark = pytest.mark.gpu


def packed_docs(seed, lens, dim, dtype):
    cu = np.zeros(len(lens) + 1, np.int64)
    np.cumsum(lens, out=cu[1:])
    D = datagen.gaussian_rows(seed, 2, int(cu[-1]), dim, dtype)
    return D, cu


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_varlen_ragged_with_empty_docs(dtype):
    lens = np.array([0, 33, 1, 300, 0, 0, 128, 129, 5, 0, 260, 31, 32, 0])
    Nq, Lq, dim = 3, 32, 128
    D, cu = packed_docs(11, lens, dim, dtype)
    Q = datagen.gaussian_rows(11, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    dm = (np.random.default_rng(2).random(int(cu[-1])) > 0.1).astype(np.uint8)
    for d_mask in (None, dm):
        s, a = ops.maxsim_fwd_varlen(dev_bits(Q, dtype), None, Lq, dev_bits(D, dtype), dev(cu.astype(np.int32)),
                                     d_mask=dev(d_mask), want_argmax=True)
        assert ops.device_status() == 0
        q_off = np.arange(Nq + 1) * Lq
        ref_s, ref_a, gap = oracle.fwd_packed(Q.reshape(-1, dim), q_off, D, cu, dtype, d_mask=d_mask)
        assert_scores(s, ref_s, Lq)
        assert_argmax(a, ref_a, gap)
        assert (s.cpu().numpy()[:, lens == 0] == 0).all()


def test_varlen_packed_queries():
    dtype, dim = "f16", 64
    qlens = np.array([5, 32, 1, 70, 17])
    dlens = np.array([40, 200, 0, 129, 7, 64])
    rng = np.random.default_rng(9)
    cu_q = np.concatenate([[0], np.cumsum(qlens)])
    cu_d = np.concatenate([[0], np.cumsum(dlens)])
    Q = datagen.float_to_bits(integer_rows(rng, int(cu_q[-1]), dim), dtype)
    D = datagen.float_to_bits(integer_rows(rng, int(cu_d[-1]), dim), dtype)
    qm = (rng.random(int(cu_q[-1])) > 0.2).astype(np.uint8)
    max_lq = int(qlens.max())
    s, a = ops.maxsim_fwd_varlen(dev_bits(Q, dtype), dev(cu_q.astype(np.int32)), max_lq, dev_bits(D, dtype),
                                 dev(cu_d.astype(np.int32)), q_mask=dev(qm), want_argmax=True)
    assert ops.device_status() == 0
    ref_s, ref_a, _ = oracle.fwd_packed(Q, cu_q, D, cu_d, dtype, q_mask=qm, lq_stride=max_lq)
    assert np.array_equal(s.cpu().numpy().astype(np.float64), ref_s)   # integer inputs: exact
    assert np.array_equal(a.cpu().numpy(), ref_a)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_varlen_every_tail_length_exact(dtype):
    # documents of 1..140 tokens: every MMA width from 16 to 128 and every
    # padding amount inside the last 16-column group; integer inputs are exact
    dim, Nq, Lq = 32, 2, 32
    lens = np.arange(1, 141)
    rng = np.random.default_rng(3)
    cu = np.concatenate([[0], np.cumsum(lens)])
    Q = datagen.float_to_bits(integer_rows(rng, Nq * Lq, dim), dtype).reshape(Nq, Lq, dim)
    D = datagen.float_to_bits(integer_rows(rng, int(cu[-1]), dim), dtype)
    dm = (rng.random(int(cu[-1])) > 0.15).astype(np.uint8)
    for d_mask in (None, dm):
        s, a = ops.maxsim_fwd_varlen(dev_bits(Q, dtype), None, Lq, dev_bits(D, dtype), dev(cu.astype(np.int32)),
                                     d_mask=dev(d_mask), want_argmax=True)
        assert ops.device_status() == 0
        ref_s, ref_a, _ = oracle.fwd_packed(Q.reshape(-1, dim), np.arange(Nq + 1) * Lq, D, cu, dtype, d_mask=d_mask)
        assert np.array_equal(s.cpu().numpy().astype(np.float64), ref_s)
        assert np.array_equal(a.cpu().numpy(), ref_a)


@pytest.mark.parametrize("dim", [128, 64])
def test_varlen_two_row_blocks_every_tail_length_exact(dim):
    # 32 queries x 32 tokens = 1024 rows (two row blocks, as in ColBERT
    # reranking) against documents of 1..140 tokens
    dtype, Nq, Lq = "f16", 32, 32
    lens = np.concatenate([np.arange(1, 141), [0, 300, 0]])
    rng = np.random.default_rng(5)
    cu = np.concatenate([[0], np.cumsum(lens)])
    Q = datagen.float_to_bits(integer_rows(rng, Nq * Lq, dim), dtype).reshape(Nq, Lq, dim)
    D = datagen.float_to_bits(integer_rows(rng, int(cu[-1]), dim), dtype)
    dm = (rng.random(int(cu[-1])) > 0.15).astype(np.uint8)
    for d_mask in (None, dm):
        s, a = ops.maxsim_fwd_varlen(dev_bits(Q, dtype), None, Lq, dev_bits(D, dtype), dev(cu.astype(np.int32)),
                                     d_mask=dev(d_mask), want_argmax=True)
        assert ops.device_status() == 0
        ref_s, ref_a, _ = oracle.fwd_packed(Q.reshape(-1, dim), np.arange(Nq + 1) * Lq, D, cu, dtype, d_mask=d_mask)
        assert np.array_equal(s.cpu().numpy().astype(np.float64), ref_s)
        assert np.array_equal(a.cpu().numpy(), ref_a)


@pytest.mark.parametrize("Lq", [32, 8, 1])
def test_varlen_many_tiny_documents_exact(Lq):
    # runs of 0..3-token documents (more than 32 document ends inside one
    # 128-row tile), then long ones; scores with and without the argmax, and
    # the argmax, exact on integer inputs (first index among equal maxima)
    dtype, dim, Nq = "f16", 64, 5
    rng = np.random.default_rng(21 + Lq)
    lens = np.concatenate([rng.integers(0, 4, 300), [0, 0, 129, 1, 0, 255], rng.integers(1, 3, 70), [128, 2, 0]])
    cu = np.concatenate([[0], np.cumsum(lens)])
    Q = datagen.float_to_bits(integer_rows(rng, Nq * Lq, dim), dtype).reshape(Nq, Lq, dim)
    D = datagen.float_to_bits(integer_rows(rng, int(cu[-1]), dim), dtype)
    dm = (rng.random(int(cu[-1])) > 0.3).astype(np.uint8)
    for d_mask in (None, dm):
        args = (dev_bits(Q, dtype), None, Lq, dev_bits(D, dtype), dev(cu.astype(np.int32)))
        s, a = ops.maxsim_fwd_varlen(*args, d_mask=dev(d_mask), want_argmax=True)
        s0, _ = ops.maxsim_fwd_varlen(*args, d_mask=dev(d_mask))
        assert ops.device_status() == 0
        ref_s, ref_a, _ = oracle.fwd_packed(Q.reshape(-1, dim), np.arange(Nq + 1) * Lq, D, cu, dtype, d_mask=d_mask)
        assert np.array_equal(s.cpu().numpy().astype(np.float64), ref_s)
        assert np.array_equal(s0.cpu().numpy().astype(np.float64), ref_s)
        assert np.array_equal(a.cpu().numpy(), ref_a)


def test_varlen_equals_dense_with_trailing_mask():
    # "same as the padded path": a trailing d_mask equals shorter packed documents
    dtype, Nq, Lq, Nd, Ld, dim = "bf16", 2, 32, 5, 200, 128
    Q = datagen.gaussian_rows(6, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(6, 2, Nd * Ld, dim, dtype).reshape(Nd, Ld, dim)
    lens = np.array([200, 150, 0, 1, 77])
    dm = (np.arange(Ld)[None, :] < lens[:, None]).astype(np.uint8)
    s_dense, a_dense = ops.maxsim_fwd(dev_bits(Q, dtype), dev_bits(D, dtype), None, dev(dm), want_argmax=True)
    packed = np.concatenate([D[j, :lens[j]] for j in range(Nd)])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    s_var, a_var = ops.maxsim_fwd_varlen(dev_bits(Q, dtype), None, Lq, dev_bits(packed, dtype), dev(cu),
                                         want_argmax=True)
    assert ops.device_status() == 0
    assert torch.equal(a_dense, a_var)
    assert torch.allclose(s_dense, s_var, rtol=0, atol=1e-5)


def test_bad_cu_seqlens_reported_on_device():
    dim = 16
    D = dev_bits(datagen.gaussian_rows(1, 2, 50, dim, "f16"), "f16")
    Q = dev_bits(datagen.gaussian_rows(1, 1, 4, dim, "f16").reshape(1, 4, dim), "f16")
    cu = dev(np.array([0, 30, 20, 50], np.int32))  # decreasing: invalid
    ops.maxsim_fwd_varlen(Q, None, 4, D, cu)
    assert ops.device_status() == 6
    assert ops.device_status() == 0  # reading clears it


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_backward_parity(dtype):
    Nq, Lq, Nd, Ld, dim = 5, 24, 6, 300, 128
    seed = 31
    Q = datagen.gaussian_rows(seed, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(seed, 2, Nd * Ld, dim, dtype).reshape(Nd, Ld, dim)
    qm = datagen.mask_drop_tail(seed, 4, Nq, Lq, 8)
    dm = np.ones((Nd, Ld), np.uint8)
    dm[2] = 0  # sentinel sources
    g = datagen.normal_f32(seed, 6, Nq * Nd).reshape(Nq, Nd)
    Qd, Dd = dev_bits(Q, dtype), dev_bits(D, dtype)
    _, a = ops.maxsim_fwd(Qd, Dd, dev(qm), dev(dm), want_argmax=True)
    dQ, dD, rp, col = ops.maxsim_bwd(Qd, Dd, a, dev(g), dev(qm), want_csr=True)
    assert ops.device_status() == 0
    am = a.cpu().numpy()
    ref_dQ, ref_dD, ref_rp, ref_col = oracle.bwd(Q, D, dtype, am, g, q_mask=qm)
    assert np.array_equal(rp.cpu().numpy(), ref_rp)
    assert np.array_equal(col.cpu().numpy()[: ref_rp[-1]], ref_col)
    assert_grad(dQ, ref_dQ)
    assert_grad(dD, ref_dD)
    # bitwise reproducible (no atomics)
    dQ2, dD2, rp2, col2 = ops.maxsim_bwd(Qd, Dd, a, dev(g), dev(qm), want_csr=True)
    n_src = int(ref_rp[-1])  # only the first row_ptr[-1] entries of col are written
    assert torch.equal(dQ, dQ2) and torch.equal(dD, dD2) and torch.equal(rp, rp2)
    assert torch.equal(col[:n_src], col2[:n_src])


def test_backward_hot_token_contention():
    # every query token of every query picks the same document token
    Nq, Lq, Nd, Ld, dim = 16, 32, 2, 64, 32
    rng = np.random.default_rng(4)
    Q = datagen.float_to_bits(np.abs(integer_rows(rng, Nq * Lq, dim)), "bf16").reshape(Nq, Lq, dim)
    Dv = np.zeros((Nd * Ld, dim))
    Dv[::Ld] = 1.0  # token 0 of each document dominates
    D = datagen.float_to_bits(Dv, "bf16").reshape(Nd, Ld, dim)
    g = datagen.normal_f32(2, 6, Nq * Nd).reshape(Nq, Nd)
    Qd, Dd = dev_bits(Q, "bf16"), dev_bits(D, "bf16")
    _, a = ops.maxsim_fwd(Qd, Dd, want_argmax=True)
    dQ, dD, rp, col = ops.maxsim_bwd(Qd, Dd, a, dev(g), want_csr=True)
    am = a.cpu().numpy()
    ref_dQ, ref_dD, ref_rp, ref_col = oracle.bwd(Q, D, "bf16", am, g)
    assert np.array_equal(rp.cpu().numpy(), ref_rp) and np.array_equal(col.cpu().numpy()[: ref_rp[-1]], ref_col)
    assert_grad(dQ, ref_dQ)
    assert_grad(dD, ref_dD)


@pytest.mark.parametrize("shape", [(5, 24, 6, 300, 128), (16, 32, 3, 64, 32), (2, 40, 4, 1030, 256),
                                   (64, 128, 2, 1024, 128)])
def test_backward_without_csr_equals_csr_path(shape):
    # Without the CSR outputs, dD comes from the shared-memory CSR of each
    # document slice: the same sources in the same order, so the same bits.
    Nq, Lq, Nd, Ld, dim = shape
    seed = 41
    Q = datagen.gaussian_rows(seed, 1, Nq * Lq, dim, "bf16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(seed, 2, Nd * Ld, dim, "bf16").reshape(Nd, Ld, dim)
    qm = datagen.mask_drop_tail(seed, 4, Nq, Lq, 8)
    dm = np.ones((Nd, Ld), np.uint8)
    dm[-1, 5:] = 0  # one document's winners crowd into its first tokens
    g = datagen.normal_f32(seed, 6, Nq * Nd).reshape(Nq, Nd)
    Qd, Dd = dev_bits(Q, "bf16"), dev_bits(D, "bf16")
    _, a = ops.maxsim_fwd(Qd, Dd, dev(qm), dev(dm), want_argmax=True)
    dQ1, dD1, _, _ = ops.maxsim_bwd(Qd, Dd, a, dev(g), dev(qm), want_csr=True)
    dQ2, dD2, _, _ = ops.maxsim_bwd(Qd, Dd, a, dev(g), dev(qm))
    _, dD3, _, _ = ops.maxsim_bwd(Qd, Dd, a, dev(g), dev(qm), want_dq=False)
    assert ops.device_status() == 0
    assert torch.equal(dD1, dD2) and torch.equal(dD2, dD3) and torch.equal(dQ1, dQ2)
    am = a.cpu().numpy()
    ref_dQ, ref_dD, _, _ = oracle.bwd(Q, D, "bf16", am, g, q_mask=qm)
    assert_grad(dQ2, ref_dQ)
    assert_grad(dD2, ref_dD)


@pytest.mark.parametrize("Nq", [128, 129])
def test_backward_shared_memory_csr_size_limit(Nq):
    # 128 x 128 = 16,384 sources per document is the largest the shared-memory
    # CSR takes; 129 queries fall back to the CSR in global memory. Both match
    # the oracle and the path that returns the CSR, bit for bit.
    Lq, Nd, Ld, dim = 128, 2, 64, 64
    seed = 43
    Q = datagen.gaussian_rows(seed, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(seed, 2, Nd * Ld, dim, "f16").reshape(Nd, Ld, dim)
    g = datagen.normal_f32(seed, 6, Nq * Nd).reshape(Nq, Nd)
    Qd, Dd = dev_bits(Q, "f16"), dev_bits(D, "f16")
    _, a = ops.maxsim_fwd(Qd, Dd, want_argmax=True)
    dQ, dD, _, _ = ops.maxsim_bwd(Qd, Dd, a, dev(g))
    dQ_c, dD_c, _, _ = ops.maxsim_bwd(Qd, Dd, a, dev(g), want_csr=True)
    assert ops.device_status() == 0
    assert torch.equal(dD, dD_c) and torch.equal(dQ, dQ_c)
    ref_dQ, ref_dD, _, _ = oracle.bwd(Q, D, "f16", a.cpu().numpy(), g)
    assert_grad(dQ, ref_dQ)
    assert_grad(dD, ref_dD)


def test_backward_side_stream_ordered_with_callers_stream():
    # dQ runs on a stream of the library's own beside the caller's: the gradient
    # written on the caller's stream just before each call, and the outputs read
    # on it just after, must be ordered with it (the stream is kept busy first,
    # so a missing fork or join would read or return stale data)
    Nq, Lq, Nd, Ld, dim = 16, 32, 6, 200, 64
    seed = 47
    Q = datagen.gaussian_rows(seed, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(seed, 2, Nd * Ld, dim, "f16").reshape(Nd, Ld, dim)
    g = datagen.normal_f32(seed, 6, Nq * Nd).reshape(Nq, Nd)
    Qd, Dd = dev_bits(Q, "f16"), dev_bits(D, "f16")
    _, a = ops.maxsim_fwd(Qd, Dd, want_argmax=True)
    g_base = dev(g)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = []
    with torch.cuda.stream(s):
        for rep in range(3):
            busy = torch.empty(64 << 20, device="cuda").uniform_()
            gr = g_base * float(rep + 1) + busy[:1] * 0.0
            dQ, dD, _, _ = ops.maxsim_bwd(Qd, Dd, a, gr)
            out.append((dQ.clone(), dD.clone()))
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    am = a.cpu().numpy()
    for rep, (dQ, dD) in enumerate(out):
        ref_dQ, ref_dD, _, _ = oracle.bwd(Q, D, "f16", am, g * float(rep + 1))
        assert_grad(dQ, ref_dQ)
        assert_grad(dD, ref_dD)


def test_backward_without_csr_hot_token():
    # every query token picks token 0 of its document: one destination row gets all sources
    Nq, Lq, Nd, Ld, dim = 64, 128, 2, 300, 64
    rng = np.random.default_rng(9)
    Q = datagen.float_to_bits(np.abs(integer_rows(rng, Nq * Lq, dim)), "bf16").reshape(Nq, Lq, dim)
    Dv = np.zeros((Nd * Ld, dim))
    Dv[::Ld] = 1.0
    D = datagen.float_to_bits(Dv, "bf16").reshape(Nd, Ld, dim)
    g = datagen.normal_f32(3, 6, Nq * Nd).reshape(Nq, Nd)
    Qd, Dd = dev_bits(Q, "bf16"), dev_bits(D, "bf16")
    _, a = ops.maxsim_fwd(Qd, Dd, want_argmax=True)
    _, dD, _, _ = ops.maxsim_bwd(Qd, Dd, a, dev(g))
    _, dD_csr, _, _ = ops.maxsim_bwd(Qd, Dd, a, dev(g), want_csr=True)
    assert ops.device_status() == 0
    assert torch.equal(dD, dD_csr)
    ref_dQ, ref_dD, _, _ = oracle.bwd(Q, D, "bf16", a.cpu().numpy(), g)
    assert_grad(dD, ref_dD)


def test_backward_without_csr_out_of_range_reported():
    Nq, Lq, Nd, Ld, dim = 1, 4, 2, 8, 16
    Q = dev_bits(datagen.gaussian_rows(1, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim), "f16")
    D = dev_bits(datagen.gaussian_rows(1, 2, Nd * Ld, dim, "f16").reshape(Nd, Ld, dim), "f16")
    a = dev(np.array([[0, 1, 9, -1], [2, 3, 4, -7]], np.int32))
    g = dev(np.ones((Nq, Nd), np.float32))
    _, dD, _, _ = ops.maxsim_bwd(Q, D, a, g)
    assert ops.device_status() == 6
    # the valid sources still land: rows 0, 1 of document 0 and 2, 3, 4 of document 1
    got = dD.cpu().numpy()
    q = datagen.bits_to_float(datagen.gaussian_rows(1, 1, Nq * Lq, dim, "f16"), "f16")
    np.testing.assert_allclose(got[0, 0], q[0], rtol=1e-6)
    np.testing.assert_allclose(got[1, 4], q[2], rtol=1e-6)
    assert not got[0, 2:].any()


def test_backward_out_of_range_argmax_reported():
    Nq, Lq, Nd, Ld, dim = 1, 4, 2, 8, 16
    Q = dev_bits(datagen.gaussian_rows(1, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim), "f16")
    D = dev_bits(datagen.gaussian_rows(1, 2, Nd * Ld, dim, "f16").reshape(Nd, Ld, dim), "f16")
    a = dev(np.array([[0, 1, 9, -1], [2, 3, 4, -7]], np.int32))
    g = dev(np.ones((Nq, Nd), np.float32))
    ops.maxsim_bwd(Q, D, a, g, want_csr=True)
    assert ops.device_status() == 6


def test_autograd_wrapper():
    from maxsim_scoring_gb300 import maxsim
    Nq, Lq, Nd, Ld, dim = 3, 16, 4, 90, 64
    Qb = datagen.gaussian_rows(2, 1, Nq * Lq, dim, "bf16").reshape(Nq, Lq, dim)
    Db = datagen.gaussian_rows(2, 2, Nd * Ld, dim, "bf16").reshape(Nd, Ld, dim)
    Q = dev_bits(Qb, "bf16").requires_grad_()
    D = dev_bits(Db, "bf16").requires_grad_()
    g = datagen.normal_f32(2, 6, Nq * Nd).reshape(Nq, Nd)
    s = maxsim(Q, D)
    (s * dev(g)).sum().backward()
    ref_s, ref_a, gap = oracle.fwd_dense(Qb, Db, "bf16")
    assert_scores(s.detach(), ref_s, Lq)
    # the gradient through the argmax the forward saved (the same call, deterministic)
    _, a = ops.maxsim_fwd(Q.detach(), D.detach(), want_argmax=True)
    am = a.cpu().numpy()
    assert_argmax(a, ref_a, gap)
    ref_dQ, ref_dD, _, _ = oracle.bwd(Qb, Db, "bf16", am, g)
    # the wrapper returns the gradients in the inputs' type (bf16)
    assert_grad_rounded(Q.grad, ref_dQ, "bf16")
    assert_grad_rounded(D.grad, ref_dD, "bf16")
