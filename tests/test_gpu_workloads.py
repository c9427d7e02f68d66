"""The five workloads at their full sizes, through the same entry points and
launch configurations the benchmark uses, checked against the CPU oracle on
seeded samples of documents (the oracle computes each sampled output on its
own) and, where it is cheap, in full."""
import numpy as np
import pytest
import torch

import oracle
from datagen import workloads
from maxsim_scoring_gb300 import ops
from tests.gpu_util import assert_argmax, assert_grad, assert_scores, dev, dev_bits

pytestmark = pytest.mark.gpu


def sample_docs(nd, n, seed):
    return np.sort(np.random.default_rng(seed).choice(nd, size=min(n, nd), replace=False))


def test_tiny_rerank_full():
    w = workloads.make("tiny_rerank")
    s, a = ops.maxsim_fwd(dev_bits(w["Q"], "f16"), dev_bits(w["D"], "f16"), want_argmax=True)
    assert ops.device_status() == 0
    ref_s, ref_a, gap = oracle.fwd_dense(w["Q"], w["D"], "f16")
    assert_scores(s, ref_s, w["Lq"])
    assert_argmax(a, ref_a, gap)


def test_colbert_varlen_full_size_sampled():
    w = workloads.make("colbert_varlen")
    Nq, Lq, dim = w["Nq"], w["Lq"], w["dim"]
    Q, D = dev_bits(w["Q"], "f16"), dev_bits(w["D"], "f16")
    cu = dev(w["cu_seqlens_d"])
    s, _ = ops.maxsim_fwd_varlen(Q, None, Lq, D, cu)          # the benchmark's call
    s2, a = ops.maxsim_fwd_varlen(Q, None, Lq, D, cu, want_argmax=True)
    assert ops.device_status() == 0
    assert torch.equal(s, s2)
    docs = sample_docs(w["Nd"], 2000, 21)
    q_off = np.arange(Nq + 1, dtype=np.int64) * Lq
    ref_s, ref_a, gap = oracle.fwd_packed(w["Q"].reshape(-1, dim), q_off, w["D"], w["cu_seqlens_d"].astype(np.int64),
                                          "f16", docs=docs)
    assert_scores(s[:, docs], ref_s, Lq)
    got_a = a.view(Nq, w["Nd"], Lq)[:, docs].reshape(-1, Lq)
    assert_argmax(got_a, ref_a, gap)
    assert torch.isfinite(s).all()


def test_colpali_cross_full_size_sampled():
    w = workloads.make("colpali_cross")
    Nq, Lq, Nd, Ld = w["Nq"], w["Lq"], w["Nd"], w["Ld"]
    s, a = ops.maxsim_fwd(dev_bits(w["Q"], "bf16"), dev_bits(w["D"], "bf16"), dev(w["q_mask"]), dev(w["d_mask"]),
                          want_argmax=True)
    assert ops.device_status() == 0
    docs = sample_docs(Nd, 24, 22)
    ref_s, ref_a, gap = oracle.fwd_dense(w["Q"], w["D"], "bf16", q_mask=w["q_mask"], d_mask=w["d_mask"], docs=docs)
    assert_scores(s[:, docs], ref_s, Lq)
    assert_argmax(a.view(Nq, Nd, Lq)[:, docs].reshape(-1, Lq), ref_a, gap)


def test_contrastive_backward_full_size():
    w = workloads.make("contrastive_bwd")
    Nq, Lq, Nd, Ld = w["Nq"], w["Lq"], w["Nd"], w["Ld"]
    Q, D = dev_bits(w["Q"], "bf16"), dev_bits(w["D"], "bf16")
    s, a = ops.maxsim_fwd(Q, D, want_argmax=True)
    docs = sample_docs(Nd, 8, 23)
    ref_s, ref_a, gap = oracle.fwd_dense(w["Q"], w["D"], "bf16", docs=docs)
    assert_scores(s[:, docs], ref_s, Lq)
    assert_argmax(a.view(Nq, Nd, Lq)[:, docs].reshape(-1, Lq), ref_a, gap)
    g = w["grad"]
    dQ, dD, rp, col = ops.maxsim_bwd(Q, D, a, dev(g), want_csr=True)
    assert ops.device_status() == 0
    am = a.cpu().numpy()
    ref_dQ, ref_dD, ref_rp, ref_col = oracle.bwd(w["Q"], w["D"], "bf16", am, g)
    assert np.array_equal(rp.cpu().numpy(), ref_rp)
    assert np.array_equal(col.cpu().numpy()[: ref_rp[-1]], ref_col)
    assert_grad(dQ, ref_dQ)
    assert_grad(dD, ref_dD)


def test_int8_rerank_full_size_sampled():
    w = workloads.make("int8_rerank")
    Nq, Lq, Nd = w["Nq"], w["Lq"], w["Nd"]
    s, a, win = ops.maxsim_fwd_int8(dev(w["Q"]), dev(w["q_scale"]), dev(w["D"]), dev(w["d_scale"]), want_win_dot=True)
    s_only, _, _ = ops.maxsim_fwd_int8(dev(w["Q"]), dev(w["q_scale"]), dev(w["D"]), dev(w["d_scale"]))
    assert ops.device_status() == 0
    assert torch.equal(s, s_only)
    docs = sample_docs(Nd, 200, 24)
    ref_s, ref_a, ref_w, gap = oracle.fwd_int8(w["Q"], w["q_scale"], w["D"], w["d_scale"], docs=docs)
    assert_scores(s[:, docs], ref_s, Lq)
    got_a = a.view(Nq, Nd, Lq)[:, docs].reshape(-1, Lq)
    assert_argmax(got_a, ref_a, gap)
    got_w = win.view(Nq, Nd, Lq)[:, docs].reshape(-1, Lq).cpu().numpy()
    same = got_a.cpu().numpy() == ref_a
    assert np.array_equal(got_w[same], ref_w[same])
