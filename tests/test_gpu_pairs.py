"""Parity of the pair-list forward (maxsim_score_pairs_packed) with the CPU
oracle: every pair's score and argmax row against the oracle's entry for its
(query, document)."""
import numpy as np
import pytest
import torch

import datagen
import oracle
from datagen import workloads
from maxsim_scoring_gb300 import ops
from tests.gpu_util import assert_argmax, assert_scores, dev, dev_bits, integer_rows

pytestmark = pytest.mark.gpu


def oracle_pairs(Q, cu_q, D, cu_d, dtype, pairs, lq_stride, q_mask=None, d_mask=None):
    """The oracle's (score, argmax row, gap row) of every pair: one oracle call
    over the documents the pairs name, then a lookup per pair."""
    docs = np.unique(pairs[:, 1])
    col = {int(j): c for c, j in enumerate(docs)}
    s, a, g = oracle.fwd_packed(Q, cu_q, D, cu_d, dtype, q_mask=q_mask, d_mask=d_mask, docs=docs, lq_stride=lq_stride)
    n_sel = len(docs)
    rows = np.array([int(i) * n_sel + col[int(j)] for i, j in pairs], dtype=np.int64)
    return (s[pairs[:, 0], [col[int(j)] for j in pairs[:, 1]]], a[rows], g[rows])


def packed(seed, lens, dim, dtype, tid):
    cu = np.zeros(len(lens) + 1, np.int64)
    np.cumsum(lens, out=cu[1:])
    return datagen.gaussian_rows(seed, tid, int(cu[-1]), dim, dtype), cu


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_random_pairs_with_empty_docs_and_duplicates(dtype):
    rng = np.random.default_rng(31)
    qlens = np.array([5, 32, 1, 40, 17, 0, 64])
    dlens = rng.integers(0, 301, size=60)
    dlens[::9] = 0
    dim = 128
    Q, cu_q = packed(31, qlens, dim, dtype, 1)
    D, cu_d = packed(31, dlens, dim, dtype, 2)
    pairs = np.stack([rng.integers(0, len(qlens), 500), rng.integers(0, len(dlens), 500)], axis=1).astype(np.int32)
    pairs[10] = pairs[3]  # a duplicate pair
    max_lq = int(qlens.max())
    s, a = ops.maxsim_score_pairs_packed(dev_bits(Q, dtype), dev(cu_q.astype(np.int32)), max_lq, dev_bits(D, dtype),
                                         dev(cu_d.astype(np.int32)), dev(pairs), want_argmax=True)
    assert ops.device_status() == 0
    ref_s, ref_a, gap = oracle_pairs(Q, cu_q, D, cu_d, dtype, pairs, max_lq)
    assert_scores(s, ref_s, max_lq)
    assert_argmax(a, ref_a, gap)
    assert torch.equal(s[10], s[3]) and torch.equal(a[10], a[3])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_inputs_with_masks_exact(dtype):
    rng = np.random.default_rng(37)
    qlens = np.array([32, 7, 128, 33])
    dlens = np.array([129, 1, 0, 300, 64, 17, 128, 255])
    dim = 64
    cu_q = np.concatenate([[0], np.cumsum(qlens)])
    cu_d = np.concatenate([[0], np.cumsum(dlens)])
    Q = datagen.float_to_bits(integer_rows(rng, int(cu_q[-1]), dim), dtype)
    D = datagen.float_to_bits(integer_rows(rng, int(cu_d[-1]), dim), dtype)
    qm = (rng.random(int(cu_q[-1])) > 0.2).astype(np.uint8)
    dm = (rng.random(int(cu_d[-1])) > 0.2).astype(np.uint8)
    pairs = np.array([[i, j] for i in range(len(qlens)) for j in range(len(dlens)) if (i + 2 * j) % 3 != 1],
                     dtype=np.int32)
    max_lq = int(qlens.max())
    s, a = ops.maxsim_score_pairs_packed(dev_bits(Q, dtype), dev(cu_q.astype(np.int32)), max_lq, dev_bits(D, dtype),
                                         dev(cu_d.astype(np.int32)), dev(pairs), dev(qm), dev(dm), want_argmax=True)
    assert ops.device_status() == 0
    ref_s, ref_a, _ = oracle_pairs(Q, cu_q, D, cu_d, dtype, pairs, max_lq, q_mask=qm, d_mask=dm)
    assert np.array_equal(s.cpu().numpy().astype(np.float64), ref_s)
    assert np.array_equal(a.cpu().numpy(), ref_a)


def test_all_pairs_equal_the_grid():
    # the full (query, document) grid as a pair list gives the grid forward's values
    dtype, dim = "bf16", 128
    rng = np.random.default_rng(41)
    Nq, Lq = 5, 32
    dlens = rng.integers(0, 260, size=37)
    Q = datagen.gaussian_rows(41, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D, cu_d = packed(41, dlens, dim, dtype, 2)
    Qd, Dd, cud = dev_bits(Q, dtype), dev_bits(D, dtype), dev(cu_d.astype(np.int32))
    grid_s, grid_a = ops.maxsim_fwd_varlen(Qd, None, Lq, Dd, cud, want_argmax=True)
    pairs = np.array([[i, j] for j in range(len(dlens)) for i in range(Nq)], dtype=np.int32)[::-1].copy()
    s, a = ops.maxsim_score_pairs_packed(Qd, None, Lq, Dd, cud, dev(pairs), want_argmax=True)
    assert ops.device_status() == 0
    pi, pj = torch.from_numpy(pairs[:, 0]).long(), torch.from_numpy(pairs[:, 1]).long()
    assert torch.equal(s.cpu(), grid_s.cpu()[pi, pj])
    assert torch.equal(a.cpu(), grid_a.cpu().view(Nq, len(dlens), Lq)[pi, pj])


def test_out_of_range_pairs_are_reported():
    dtype, dim = "f16", 128
    Q = datagen.gaussian_rows(43, 1, 2 * 32, dim, dtype).reshape(2, 32, dim)
    dlens = np.array([50, 70, 90])
    D, cu_d = packed(43, dlens, dim, dtype, 2)
    pairs = np.array([[0, 1], [2, 0], [1, -1], [1, 2], [-3, 0], [0, 3]], dtype=np.int32)
    s, a = ops.maxsim_score_pairs_packed(dev_bits(Q, dtype), None, 32, dev_bits(D, dtype), dev(cu_d.astype(np.int32)),
                                         dev(pairs), want_argmax=True)
    assert ops.device_status() == 6  # MAXSIM_ERR_DEVICE_INPUT
    bad = np.array([False, True, True, False, True, True])
    assert (s.cpu().numpy()[bad] == 0).all() and (a.cpu().numpy()[bad] == -1).all()
    ok = pairs[~bad]
    ref_s, ref_a, gap = oracle_pairs(Q.reshape(-1, dim), np.arange(3) * 32, D, cu_d, dtype, ok, 32)
    assert_scores(s[torch.from_numpy(~bad)], ref_s, 32)
    assert_argmax(a[torch.from_numpy(~bad)], ref_a, gap)


def test_one_query_many_pairs():
    # a single query: every unit is a chunk of its pair list
    dtype, dim = "f16", 128
    rng = np.random.default_rng(47)
    dlens = rng.integers(1, 300, size=3000)
    D, cu_d = packed(47, dlens, dim, dtype, 2)
    Q = datagen.gaussian_rows(47, 1, 32, dim, dtype).reshape(1, 32, dim)
    pairs = np.stack([np.zeros(4000, np.int32), rng.integers(0, 3000, 4000).astype(np.int32)], axis=1)
    s, _ = ops.maxsim_score_pairs_packed(dev_bits(Q, dtype), None, 32, dev_bits(D, dtype), dev(cu_d.astype(np.int32)),
                                         dev(pairs))
    assert ops.device_status() == 0
    ref_s, _, _ = oracle_pairs(Q.reshape(-1, dim), np.array([0, 32]), D, cu_d, dtype, pairs, 32)
    assert_scores(s, ref_s, 32)


def test_colbert_corpus_sampled_pairs():
    # the 100,000-document packed corpus with 200,000 random pairs; a seeded
    # sample of the pairs is checked against the oracle one by one
    w = workloads.make("colbert_varlen")
    Nq, Lq, Nd, dim = w["Nq"], w["Lq"], w["Nd"], w["dim"]
    rng = np.random.default_rng(53)
    pairs = np.stack([rng.integers(0, Nq, 200_000), rng.integers(0, Nd, 200_000)], axis=1).astype(np.int32)
    s, _ = ops.maxsim_score_pairs_packed(dev_bits(w["Q"], "f16"), None, Lq, dev_bits(w["D"], "f16"),
                                         dev(w["cu_seqlens_d"]), dev(pairs))
    assert ops.device_status() == 0
    pick = np.sort(rng.choice(len(pairs), size=2000, replace=False))
    ref_s, _, _ = oracle_pairs(w["Q"].reshape(-1, dim), np.arange(Nq + 1) * Lq, w["D"],
                               w["cu_seqlens_d"].astype(np.int64), "f16", pairs[pick], Lq)
    assert_scores(s[torch.from_numpy(pick)], ref_s, Lq)
    assert torch.isfinite(s).all()
