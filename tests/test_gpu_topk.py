"""Parity of maxsim_topk and maxsim_two_stage_topk with the CPU oracle.

Selection is compared bit for bit wherever both sides select from the same
fp32 values (the top-k kernel on given scores, the INT8 stage's candidates
from the kernel's own stage-1 scores, everything on small-integer inputs).
Scores are compared with the forward's tolerance, 1e-3 * Lq; a final document
that differs from the oracle's choice must be within twice that tolerance of
the oracle's k-th score.
"""
import numpy as np
import pytest
import torch

import oracle
from datagen import workloads
from maxsim_scoring_gb300 import ops
from tests.gpu_util import assert_scores, dev, dev_bits

pytestmark = pytest.mark.gpu


def gpu_topk(s, k):
    vals, idx = ops.maxsim_topk(dev(np.ascontiguousarray(s, dtype=np.float32)), k)
    assert ops.device_status() == 0
    return idx.cpu().numpy(), vals.cpu().numpy()


@pytest.mark.parametrize("R,n,k", [(1, 1, 1), (3, 1000, 1000), (5, 100_003, 100), (2, 70_000, 4096), (4, 5000, 1),
                                   (2, 4097, 4096)])
def test_topk_matches_the_stable_order(R, n, k):
    rng = np.random.default_rng(n + k)
    s = (rng.integers(-50, 50, size=(R, n)) * 0.25).astype(np.float32)  # many ties
    s[:, ::11] = -0.0
    s[:, 5::13] = 0.0
    idx, vals = gpu_topk(s, k)
    ref_idx, ref_vals = oracle.topk(s, k)
    assert np.array_equal(idx, ref_idx)
    assert np.array_equal(vals.astype(np.float64), ref_vals)


def test_topk_continuous_values_and_infinities():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((6, 30_000)).astype(np.float32)
    s[0, 100] = np.inf
    s[1, :] = -np.inf
    s[2, 7] = np.nan  # ranks below every number
    idx, vals = gpu_topk(s, 300)
    ref = np.where(np.isnan(s), -np.inf, s)
    ref_idx, _ = oracle.topk(ref, 300)
    assert np.array_equal(idx[[0, 1, 3, 4, 5]], ref_idx[[0, 1, 3, 4, 5]])
    assert 7 not in idx[2].tolist() and np.array_equal(idx[2], ref_idx[2])
    assert np.array_equal(vals[0][:1], [np.inf])


def two_stage_inputs(seed, Nq, Lq, Nd, Ld, dim, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        q = rng.integers(-3, 4, size=(Nq, Lq, dim))
        d = rng.integers(-3, 4, size=(Nd, Ld, dim))
        import datagen
        return (q.astype(np.int8), np.ones((Nq, Lq), np.float32), d.astype(np.int8), np.ones((Nd, Ld), np.float32),
                datagen.float_to_bits(q.astype(np.float64), "f16"), datagen.float_to_bits(d.astype(np.float64), "f16"))
    w = workloads.two_stage(Nq, Lq, Nd, Ld, dim, 1, 1, seed)
    return w["Q8"], w["q_scale"], w["D8"], w["d_scale"], w["Q16"], w["D16"]


def run_two_stage(Q8, qs, D8, ds, Q16, D16, k1, k):
    top_idx, top_scores, s8, cand = ops.maxsim_two_stage_topk(dev(Q8), dev(qs), dev(D8), dev(ds), dev_bits(Q16, "f16"),
                                                              dev_bits(D16, "f16"), k1, k, want_stage1=True)
    assert ops.device_status() == 0
    return top_idx.cpu().numpy(), top_scores.cpu().numpy(), s8.cpu().numpy(), cand.cpu().numpy()


def test_two_stage_integer_inputs_exact():
    Q8, qs, D8, ds, Q16, D16 = two_stage_inputs(5, 3, 32, 700, 40, 64, integer=True)
    got = run_two_stage(Q8, qs, D8, ds, Q16, D16, 150, 25)
    ref = oracle.two_stage_topk(Q8, qs, D8, ds, Q16, D16, "f16", 150, 25)
    top_idx, top_scores, s8, cand = got
    assert np.array_equal(s8.astype(np.float64), ref[2])
    assert np.array_equal(cand, ref[3])
    assert np.array_equal(top_idx, ref[0]) and np.array_equal(top_scores.astype(np.float64), ref[1])


@pytest.mark.parametrize("Lq", [32, 100])
def test_two_stage_gaussian(Lq):
    Nq, Nd, Ld, dim, k1, k = 4, 3000, 64, 128, 200, 20
    Q8, qs, D8, ds, Q16, D16 = two_stage_inputs(11 + Lq, Nq, Lq, Nd, Ld, dim)
    top_idx, top_scores, s8, cand = run_two_stage(Q8, qs, D8, ds, Q16, D16, k1, k)
    # stage 1: scores against the oracle, candidates exactly from the kernel's own scores
    ref8, _, _, _ = oracle.fwd_int8(Q8, qs, D8, ds)
    assert_scores(torch.from_numpy(s8), ref8, Lq)
    cand_ref, _ = oracle.topk(s8, k1)
    assert np.array_equal(cand, cand_ref)
    # stage 2: the rescored scores of the final documents, and the selection
    exact, _, _ = oracle.fwd_dense(Q16, D16, "f16")
    tol = 1e-3 * Lq
    for i in range(Nq):
        assert set(top_idx[i].tolist()) <= set(cand[i].tolist())
        assert (np.diff(top_scores[i]) <= 0).all()
        assert np.all(np.abs(top_scores[i] - exact[i, top_idx[i]]) <= tol)
        ref_idx, ref_scores = oracle.topk(exact[i:i + 1, cand[i]], k)
        kth = ref_scores[0, -1]
        missing = set(cand[i][ref_idx[0]].tolist()) - set(top_idx[i].tolist())
        for j in missing:  # only near-ties may be swapped
            assert exact[i, j] <= kth + 2 * tol


def test_two_stage_full_corpus_sampled():
    # 32 queries over the 100,000-document corpus (k1 = 1,000, k = 100): stage-1
    # scores of a seeded sample of documents, the candidates from the kernel's own
    # scores, and two queries' final lists rescored by the oracle
    w = workloads.make("two_stage_topk")
    Lq, k1, k = w["Lq"], w["k1"], w["k"]
    top_idx, top_scores, s8, cand = run_two_stage(w["Q8"], w["q_scale"], w["D8"], w["d_scale"], w["Q16"], w["D16"],
                                                  k1, k)
    rng = np.random.default_rng(17)
    docs = np.sort(rng.choice(w["Nd"], size=200, replace=False))
    ref8, _, _, _ = oracle.fwd_int8(w["Q8"], w["q_scale"], w["D8"], w["d_scale"], docs=docs)
    assert_scores(torch.from_numpy(s8[:, docs]), ref8, Lq)
    cand_ref, _ = oracle.topk(s8, k1)
    assert np.array_equal(cand, cand_ref)
    for i in (0, 31):
        exact, _, _ = oracle.fwd_dense(w["Q16"][i:i + 1], w["D16"], "f16", docs=cand[i].astype(np.int64))
        pos = {int(j): c for c, j in enumerate(cand[i])}
        got = exact[0, [pos[int(j)] for j in top_idx[i]]]
        assert np.all(np.abs(top_scores[i] - got) <= 1e-3 * Lq)
        kth = np.sort(exact[0])[::-1][k - 1]
        assert got.min() >= kth - 2e-3 * Lq
