"""Parity of the dense forward (maxsim_fwd) with the CPU oracle."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from maxsim_scoring_gb300 import ops
from tests.gpu_util import assert_argmax, assert_scores, dev, dev_bits, integer_rows

pytestmark = pytest.mark.gpu


def run_case(Q, D, dtype, q_mask=None, d_mask=None, exact=False):
    Nq, Lq, dim = Q.shape
    s, a = ops.maxsim_fwd(dev_bits(Q, dtype), dev_bits(D, dtype), dev(q_mask), dev(d_mask), want_argmax=True)
    s_only, _ = ops.maxsim_fwd(dev_bits(Q, dtype), dev_bits(D, dtype), dev(q_mask), dev(d_mask))
    assert ops.device_status() == 0
    ref_s, ref_a, gap = oracle.fwd_dense(Q, D, dtype, q_mask=q_mask, d_mask=d_mask)
    if exact:
        assert np.array_equal(s.cpu().numpy().astype(np.float64), ref_s)
        assert np.array_equal(a.cpu().numpy(), ref_a)
    else:
        assert_scores(s, ref_s, Lq)
        assert_argmax(a, ref_a, gap)
    # the argmax-free variant computes the same scores bit for bit
    assert torch.equal(s, s_only)
    return s, a


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [
    (3, 32, 5, 300, 128),   # aligned queries, tiles spanning documents, ragged tail
    (2, 40, 4, 257, 128),   # padded queries (40 -> 64 rows)
    (5, 8, 7, 130, 64),     # several queries per warp
    (2, 17, 3, 129, 96),    # dim not a multiple of 64
    (3, 64, 3, 200, 256),   # dim > 128: two 128-wide slices accumulate before the max
])
def test_integer_inputs_bit_exact(dtype, shape):
    Nq, Lq, Nd, Ld, dim = shape
    rng = np.random.default_rng(sum(shape))
    Q = datagen.float_to_bits(integer_rows(rng, Nq * Lq, dim), dtype).reshape(Nq, Lq, dim)
    D = datagen.float_to_bits(integer_rows(rng, Nd * Ld, dim), dtype).reshape(Nd, Ld, dim)
    qm = (rng.random((Nq, Lq)) > 0.2).astype(np.uint8)
    dm = (rng.random((Nd, Ld)) > 0.2).astype(np.uint8)
    run_case(Q, D, dtype, exact=True)                 # many exact ties: lowest index must win
    run_case(Q, D, dtype, q_mask=qm, d_mask=dm, exact=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(4, 32, 6, 333, 128), (2, 128, 3, 1024, 128), (3, 7, 9, 45, 128)])
def test_gaussian_inputs(dtype, shape):
    Nq, Lq, Nd, Ld, dim = shape
    seed = 17 + sum(shape)
    Q = datagen.gaussian_rows(seed, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(seed, 2, Nd * Ld, dim, dtype).reshape(Nd, Ld, dim)
    qm = datagen.mask_drop_tail(seed, 4, Nq, Lq, max(1, Lq // 3))
    dm = datagen.mask_random_subset(seed, 5, Nd, Ld, Ld // 5)
    run_case(Q, D, dtype)
    run_case(Q, D, dtype, q_mask=qm, d_mask=dm)


def test_long_query_chunked():
    # Lq > 512 rows: the query is split into row blocks whose partial scores are summed
    Nq, Lq, Nd, Ld, dim = 2, 1100, 3, 150, 128
    Q = datagen.gaussian_rows(3, 1, Nq * Lq, dim, "bf16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(3, 2, Nd * Ld, dim, "bf16").reshape(Nd, Ld, dim)
    qm = datagen.mask_drop_tail(3, 4, Nq, Lq, 200)
    run_case(Q, D, "bf16", q_mask=qm)


def test_degenerate_shapes():
    rng = np.random.default_rng(5)
    for (Nq, Lq, Nd, Ld, dim) in [(1, 1, 1, 1, 16), (2, 1, 3, 5, 32), (1, 5, 4, 1, 64), (3, 3, 2, 2, 16)]:
        Q = datagen.float_to_bits(integer_rows(rng, Nq * Lq, dim), "f16").reshape(Nq, Lq, dim)
        D = datagen.float_to_bits(integer_rows(rng, Nd * Ld, dim), "f16").reshape(Nd, Ld, dim)
        run_case(Q, D, "f16", exact=True)


def test_fully_masked_documents_and_rows():
    Nq, Lq, Nd, Ld, dim = 2, 32, 4, 150, 128
    Q = datagen.gaussian_rows(8, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(8, 2, Nd * Ld, dim, "f16").reshape(Nd, Ld, dim)
    dm = np.ones((Nd, Ld), np.uint8)
    dm[1] = 0
    dm[3, 1:] = 0
    qm = np.ones((Nq, Lq), np.uint8)
    qm[1] = 0
    s, a = run_case(Q, D, "f16", q_mask=qm, d_mask=dm)
    s = s.cpu().numpy()
    assert (s[:, 1] == 0).all() and (s[1] == 0).all()
    assert (a.cpu().numpy().reshape(Nq, Nd, Lq)[:, 1] == -1).all()


def test_negative_scores_keep_their_max():
    # all similarities negative: a masked position must not win with 0
    Q = datagen.float_to_bits(-np.ones((1, 32, 16)), "f16")
    D = datagen.float_to_bits(np.abs(integer_rows(np.random.default_rng(1), 40, 16)) + 1, "f16").reshape(1, 40, 16)
    dm = np.ones((1, 40), np.uint8)
    dm[0, ::2] = 0
    s, _ = run_case(Q, D, "f16", d_mask=dm, exact=True)
    assert (s.cpu().numpy() < 0).all()


def test_repeatable_bitwise():
    Nq, Lq, Nd, Ld, dim = 8, 32, 50, 700, 128
    Q = dev_bits(datagen.gaussian_rows(4, 1, Nq * Lq, dim, "bf16").reshape(Nq, Lq, dim), "bf16")
    D = dev_bits(datagen.gaussian_rows(4, 2, Nd * Ld, dim, "bf16").reshape(Nd, Ld, dim), "bf16")
    first = ops.maxsim_fwd(Q, D, want_argmax=True)
    for _ in range(3):
        again = ops.maxsim_fwd(Q, D, want_argmax=True)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    assert ops.device_status() == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [
    (40, 32, 7, 300, 128),   # 1280 query rows: three row blocks
    (8, 128, 5, 260, 128),   # 1024 rows: one full pair of row blocks
    (20, 48, 4, 97, 64),     # padded queries (48 -> 64 rows), 1280 rows
    (6, 64, 3, 200, 256),    # dim 256 on the CTA pair: two 256-row blocks, four-step K chains
])
def test_several_row_blocks_integer_exact(dtype, shape):
    # more than one 512-row block of query rows; exact integers make every
    # argmax (ties included) comparable bit for bit
    Nq, Lq, Nd, Ld, dim = shape
    rng = np.random.default_rng(7 + sum(shape))
    Q = datagen.float_to_bits(integer_rows(rng, Nq * Lq, dim), dtype).reshape(Nq, Lq, dim)
    D = datagen.float_to_bits(integer_rows(rng, Nd * Ld, dim), dtype).reshape(Nd, Ld, dim)
    qm = (rng.random((Nq, Lq)) > 0.2).astype(np.uint8)
    dm = (rng.random((Nd, Ld)) > 0.2).astype(np.uint8)
    run_case(Q, D, dtype, exact=True)
    run_case(Q, D, dtype, q_mask=qm, d_mask=dm, exact=True)


def test_colpali_like_gaussian():
    Nq, Lq, Nd, Ld, dim = 16, 128, 6, 1024, 128
    Q = datagen.gaussian_rows(12, 1, Nq * Lq, dim, "bf16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(12, 2, Nd * Ld, dim, "bf16").reshape(Nd, Ld, dim)
    qm = datagen.mask_drop_tail(12, 4, Nq, Lq, 40)
    dm = datagen.mask_random_subset(12, 5, Nd, Ld, 200)
    run_case(Q, D, "bf16", q_mask=qm, d_mask=dm)
