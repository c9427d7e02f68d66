"""The five synthetic workloads of the MaxSim operator, as seeded host arrays.

Shapes and distributions follow the workloads the pages measure (ColBERT
reranking, ColPali cross products, contrastive training, INT8 visual rerank);
no dataset item is reproduced: every value is drawn from the seeded
generators in this package.

 tiny_rerank      Q [1,32,128] f16, D [1000,180,128] f16, no masks, seed 0
 colbert_varlen   Q [32,32,128] f16, D packed with cu_seqlens, Ld ~ U{32..300},
                  Nd = 100,000, seed 2
 colpali_cross    Q [128,128,128] bf16, D [128,1024,128] bf16, q_mask drops the
                  last k ~ U{0..40} query tokens, d_mask hides a random subset of
                  k ~ U{0..200} doc patches, seed 3
 contrastive_bwd  Q [64,128,128] bf16, D [64,1024,128] bf16, grad [64,64] f32
                  N(0,1), seed 4
 int8_rerank      Q int8 [1,1024,128] + scales, D int8 [10000,1024,128] + scales,
                  seed 5
 colbert_pairs    the colbert_varlen corpus and queries with 10,000 (query,
                  document) pairs per query, documents uniform over the corpus
                  (a reranker's candidate lists), seed 2
Every row is an l2-normalised Gaussian vector rounded once to its storage type.

 colbert_varlen_bwd  training-side backward on packed documents: Q [64,32,128]
                  bf16, D packed with Ld ~ U{32..300}, Nd = 4,096, grad [64,4096]
                  f32 N(0,1), seed 9
 two_stage_topk   Q [32,32,128] and D [100000,128,128] as INT8 (per-token
                  scales) and as f16: the same l2-normalised Gaussian rows
                  quantised two ways; k1 = 1,000 candidates, k = 100, seed 7
 colpali_out_of_core  one query Q [1,32,128] bf16 against a corpus of 100,000
                  documents x 1,024 patches x 128 bf16 (26 GB) held in host
                  memory and streamed in blocks of 20,000 documents, seed 8
 chamfer_100k     one pair of 3-D point clouds of 100,000 points each
                  (standard normal coordinates, float32) and an upstream
                  gradient N(0,1) per pair, seed 6: the Chamfer-distance
                  workload at the cloud size the pages run
"""
from __future__ import annotations

import numpy as np

from . import (TID_CLOUD_GRAD, TID_CLOUD_P, TID_CLOUD_Q, TID_D, TID_DMASK, TID_GRAD, TID_LEN_D, TID_PAIR_D, TID_Q,
               TID_QMASK, gaussian_rows, int8_rows, mask_drop_tail, mask_random_subset, normal_f32, uniform_int)

SPECS = {
    "tiny_rerank": dict(Nq=1, Lq=32, Nd=1000, Ld=180, dim=128, dtype="f16", seed=0),
    "colbert_varlen": dict(Nq=32, Lq=32, Nd=100_000, ld_min=32, ld_max=300, dim=128, dtype="f16", seed=2),
    "colpali_cross": dict(Nq=128, Lq=128, Nd=128, Ld=1024, dim=128, dtype="bf16", seed=3,
                          q_drop_max=40, d_hide_max=200),
    "contrastive_bwd": dict(Nq=64, Lq=128, Nd=64, Ld=1024, dim=128, dtype="bf16", seed=4),
    "int8_rerank": dict(Nq=1, Lq=1024, Nd=10_000, Ld=1024, dim=128, seed=5),
    "colbert_pairs": dict(Nq=32, Lq=32, Nd=100_000, ld_min=32, ld_max=300, dim=128, dtype="f16", seed=2,
                          pairs_per_query=10_000),
    "chamfer_100k": dict(B=1, N=100_000, M=100_000, dim=3, seed=6),
    "two_stage_topk": dict(Nq=32, Lq=32, Nd=100_000, Ld=128, dim=128, k1=1000, k=100, seed=7),
    "colbert_varlen_bwd": dict(Nq=64, Lq=32, Nd=4096, ld_min=32, ld_max=300, dim=128, dtype="bf16", seed=9),
    "colpali_out_of_core": dict(Nq=1, Lq=32, Nd=100_000, Ld=1024, dim=128, dtype="bf16", block_docs=20_000, seed=8),
}


def dense(Nq, Lq, Nd, Ld, dim, dtype, seed, q_drop_max=None, d_hide_max=None, grad=False):
    """Dense Q [Nq,Lq,dim] and D [Nd,Ld,dim] (+ optional masks / gradient)."""
    w = dict(Nq=Nq, Lq=Lq, Nd=Nd, Ld=Ld, dim=dim, dtype=dtype, seed=seed)
    w["Q"] = gaussian_rows(seed, TID_Q, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    w["D"] = gaussian_rows(seed, TID_D, Nd * Ld, dim, dtype).reshape(Nd, Ld, dim)
    w["q_mask"] = mask_drop_tail(seed, TID_QMASK, Nq, Lq, q_drop_max) if q_drop_max is not None else None
    w["d_mask"] = mask_random_subset(seed, TID_DMASK, Nd, Ld, d_hide_max) if d_hide_max is not None else None
    w["grad"] = normal_f32(seed, TID_GRAD, Nq * Nd).reshape(Nq, Nd) if grad else None
    return w


def varlen(Nq, Lq, Nd, ld_min, ld_max, dim, dtype, seed):
    """Dense Q [Nq,Lq,dim]; D packed [sum Ld, dim] with int32 cu_seqlens [Nd+1]."""
    w = dict(Nq=Nq, Lq=Lq, Nd=Nd, dim=dim, dtype=dtype, seed=seed)
    lens = uniform_int(seed, TID_LEN_D, Nd, ld_min, ld_max)
    cu = np.zeros(Nd + 1, dtype=np.int64)
    np.cumsum(lens, out=cu[1:])
    assert cu[-1] < 2**31
    w["lens"] = lens
    w["cu_seqlens_d"] = cu.astype(np.int32)
    w["total_d"] = int(cu[-1])
    w["max_ld"] = int(lens.max()) if Nd else 0
    w["Q"] = gaussian_rows(seed, TID_Q, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    w["D"] = gaussian_rows(seed, TID_D, int(cu[-1]), dim, dtype)
    return w


def pairs(Nq, Lq, Nd, ld_min, ld_max, dim, dtype, seed, pairs_per_query):
    """The varlen corpus plus int32 pairs [Nq * pairs_per_query, 2]: query i
    owns rows i * pairs_per_query ..., each naming a uniform random document."""
    w = varlen(Nq, Lq, Nd, ld_min, ld_max, dim, dtype, seed)
    n = Nq * pairs_per_query
    docs = uniform_int(seed, TID_PAIR_D, n, 0, Nd - 1) if n else np.zeros(0, np.int32)
    w["pairs"] = np.stack([np.repeat(np.arange(Nq, dtype=np.int32), pairs_per_query), docs], axis=1)
    w["num_pairs"] = n
    return w


def int8(Nq, Lq, Nd, Ld, dim, seed):
    """INT8 Q/D with one float32 scale per token (per-token symmetric)."""
    w = dict(Nq=Nq, Lq=Lq, Nd=Nd, Ld=Ld, dim=dim, seed=seed)
    q, qs = int8_rows(seed, TID_Q, Nq * Lq, dim)
    d, ds = int8_rows(seed, TID_D, Nd * Ld, dim)
    w["Q"], w["q_scale"] = q.reshape(Nq, Lq, dim), qs.reshape(Nq, Lq)
    w["D"], w["d_scale"] = d.reshape(Nd, Ld, dim), ds.reshape(Nd, Ld)
    return w


def two_stage(Nq, Lq, Nd, Ld, dim, k1, k, seed):
    """INT8 (with per-token scales) and f16 versions of the same dense Q / D:
    every row is drawn once and quantised both ways."""
    w = int8(Nq, Lq, Nd, Ld, dim, seed)
    w["Q8"], w["D8"] = w.pop("Q"), w.pop("D")
    w["Q16"] = gaussian_rows(seed, TID_Q, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim)
    w["D16"] = gaussian_rows(seed, TID_D, Nd * Ld, dim, "f16").reshape(Nd, Ld, dim)
    w.update(k1=k1, k=k, dtype="f16")
    return w


def out_of_core(Nq, Lq, Nd, Ld, dim, dtype, block_docs, seed):
    """The query batch only: the corpus is written by fill_corpus into
    caller-provided (page-locked) host memory, block by block."""
    w = dict(Nq=Nq, Lq=Lq, Nd=Nd, Ld=Ld, dim=dim, dtype=dtype, block_docs=block_docs, seed=seed)
    w["Q"] = gaussian_rows(seed, TID_Q, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    return w


def fill_corpus(w, out, chunk_docs=4096):
    """Document rows of an out-of-core workload into out (uint16 [Nd*Ld, dim])."""
    rows = w["Ld"] * chunk_docs
    for r0 in range(0, w["Nd"] * w["Ld"], rows):
        n = min(rows, w["Nd"] * w["Ld"] - r0)
        gaussian_rows(w["seed"], TID_D, n, w["dim"], w["dtype"], row0=r0, out=out[r0:r0 + n])
    return out


def clouds(B, N, M, dim, seed):
    """Point clouds P [B,N,dim], Q [B,M,dim] (float32, standard normal
    coordinates) and an upstream gradient grad [B] (float32, N(0,1))."""
    w = dict(B=B, N=N, M=M, dim=dim, seed=seed)
    w["P"] = gaussian_rows(seed, TID_CLOUD_P, B * N, dim, "f32", normalize=False).reshape(B, N, dim)
    w["Q"] = gaussian_rows(seed, TID_CLOUD_Q, B * M, dim, "f32", normalize=False).reshape(B, M, dim)
    w["grad"] = normal_f32(seed, TID_CLOUD_GRAD, B)
    return w


def make(name: str, **overrides):
    """Build a named workload; keyword overrides shrink it for quick tests."""
    spec = dict(SPECS[name])
    spec.update(overrides)
    if name == "colbert_varlen":
        return varlen(**spec)
    if name == "colbert_pairs":
        return pairs(**spec)
    if name == "colbert_varlen_bwd":
        w = varlen(**spec)
        w["grad"] = normal_f32(spec["seed"], TID_GRAD, w["Nq"] * w["Nd"]).reshape(w["Nq"], w["Nd"])
        return w
    if name == "int8_rerank":
        return int8(**spec)
    if name == "chamfer_100k":
        return clouds(**spec)
    if name == "two_stage_topk":
        return two_stage(**spec)
    if name == "colpali_out_of_core":
        return out_of_core(**spec)
    grad = name == "contrastive_bwd"
    return dense(**spec, grad=grad)
