"""Every document of the two large workloads, checked bit for bit.

The operator is exact ("Flash-MaxSim" paper, Sec. 4.1.1: the fused result is
the same computation as the offline one). With small-integer embeddings every
product and every fp32 partial sum the kernels form is an exact integer (or an
exact multiple of a power of two), so the order of the additions cannot matter
and the GPU must equal the CPU oracle exactly on every score and every argmax,
ties included (lowest index). Shapes, document-length mix and launch
configuration are those of the ColBERT varlen rerank (32 x 32 query tokens,
100,000 packed documents of U{32..300} tokens, dim 128, f16) and of the INT8
visual rerank (1 x 1024 query tokens in 512-row chunks, 10,000 x 1024 document
tokens, dim 128, per-token scales)."""
import numpy as np
import pytest
import torch

import oracle
from datagen import workloads
from maxsim_scoring_gb300 import ops
from tests.gpu_util import dev, dev_bits

pytestmark = pytest.mark.gpu


def _small_int_f16_bits(rng, shape, lo, hi):
    """Integers in [lo, hi] as binary16 bit patterns (every such integer is exact)."""
    table = np.arange(lo, hi + 1, dtype=np.float16).view(np.uint16)
    return np.take(table, rng.integers(0, hi - lo + 1, size=shape, dtype=np.int8))


def test_colbert_varlen_every_document_integer_exact():
    w = workloads.make("colbert_varlen")  # the length mix and offsets of the workload
    Nq, Lq, Nd, dim = w["Nq"], w["Lq"], w["Nd"], w["dim"]
    cu = w["cu_seqlens_d"]
    total = int(cu[-1])
    rng = np.random.default_rng(2024)
    # |<q, d>| <= 3 * 3 * 128 and a score <= 32 of those: every fp32 sum is exact
    Qb = _small_int_f16_bits(rng, (Nq * Lq, dim), -3, 3)
    Db = _small_int_f16_bits(rng, (total, dim), -3, 3)
    Q, D, cud = dev_bits(Qb.reshape(Nq, Lq, dim), "f16"), dev_bits(Db, "f16"), dev(cu)
    s, _ = ops.maxsim_fwd_varlen(Q, None, Lq, D, cud)  # the benchmark's call
    s2, a = ops.maxsim_fwd_varlen(Q, None, Lq, D, cud, want_argmax=True)
    assert ops.device_status() == 0
    del D
    ref_s, ref_a, _ = oracle.fwd_packed(Qb, np.arange(Nq + 1, dtype=np.int64) * Lq, Db, cu.astype(np.int64), "f16")
    got = s.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref_s), f"{(got != ref_s).sum()} of {got.size} scores differ"
    assert torch.equal(s, s2)
    got_a = a.cpu().numpy()
    assert np.array_equal(got_a, ref_a), f"{(got_a != ref_a).sum()} argmax entries differ"


def test_int8_rerank_every_document_integer_exact():
    w = workloads.make("int8_rerank")
    Nq, Lq, Nd, Ld, dim = w["Nq"], w["Lq"], w["Nd"], w["Ld"], w["dim"]
    rng = np.random.default_rng(2025)
    Q8 = rng.integers(-4, 5, size=(Nq, Lq, dim), dtype=np.int8)
    D8 = rng.integers(-4, 5, size=(Nd, Ld, dim), dtype=np.int8)
    # power-of-two scales: dot * d_scale and q_scale * m are exact in fp32
    pow2 = np.array([0.5, 1.0, 2.0], np.float32)
    qs = pow2[rng.integers(0, 3, size=(Nq, Lq))]
    ds = pow2[rng.integers(0, 3, size=(Nd, Ld))]
    s, a, win = ops.maxsim_fwd_int8(dev(Q8), dev(qs), dev(D8), dev(ds), want_win_dot=True)
    s_only, _, _ = ops.maxsim_fwd_int8(dev(Q8), dev(qs), dev(D8), dev(ds))  # the benchmark's call
    assert ops.device_status() == 0
    ref_s, ref_a, ref_w, _ = oracle.fwd_int8(Q8, qs, D8, ds)
    # Precondition of exactness: every value is a multiple of 1/4 and the
    # magnitudes of the terms of a score sum to below 2^22, so every fp32
    # partial sum (in any order, chunked or not) is exact.
    m = ref_w.astype(np.float64) * np.take_along_axis(np.broadcast_to(ds, (Nq, Nd, Ld)).reshape(Nq * Nd, Ld),
                                                      np.maximum(ref_a, 0), axis=1)
    assert (np.abs(m * np.repeat(qs, Nd, axis=0)).sum(axis=1) < 2.0 ** 22).all()
    got = s.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref_s), f"{(got != ref_s).sum()} of {got.size} scores differ"
    assert torch.equal(s, s_only)
    assert np.array_equal(a.cpu().numpy(), ref_a)
    assert np.array_equal(win.cpu().numpy(), ref_w)
