"""Parity of the Chamfer distance kernels (maxsim_chamfer_fwd / _bwd) with the
CPU oracle ("Flash-MaxSim" Sec. 4.2.4).

Nearest indices: the kernels search on the shifted value ||y||^2 - 2<x,y>, the
oracle in double on sum_k (x_k - y_k)^2. Where both are exact (small integer
coordinates, or coordinates on a coarse grid) the indices must be identical,
ties included (lowest index). Elsewhere an index that differs from the
oracle's must still be a nearest point within the error bound e(x, y) of the
search value:
    d(x, y_gpu) <= d(x, y_oracle) + e(x, y_gpu) + e(x, y_oracle).
 * dim > 4, fp32 FMA chain: e = 8 u (|x|^2 + |y|^2), u = 2^-24 (one rounding
   for each of dim + 2 operations whose partial values are bounded by
   |x|^2 + |y|^2 + 2|<x,y>| <= 2 (|x|^2 + |y|^2)).
 * dim <= 4, tensor cores with the two-part tf32 split: the dropped low-part
   products and the rounding of the low parts are below 3 * 2^-22 * 2|x||y|,
   and the fp32 accumulation of at most 16 products, each partial sum below
   2 (|x|^2 + |y|^2), adds at most 16 * 2^-23 of that: e = 2^-17 (|x|^2 + |y|^2).
"""
import numpy as np
import pytest
import torch

import oracle
from datagen import workloads
from maxsim_scoring_gb300 import chamfer_distance, ops
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def clouds(seed, B, N, M, dim, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        P = rng.integers(-6, 7, size=(B, N, dim)).astype(np.float32)
        Q = rng.integers(-6, 7, size=(B, M, dim)).astype(np.float32)
    else:
        P = rng.standard_normal((B, N, dim)).astype(np.float32)
        Q = rng.standard_normal((B, M, dim)).astype(np.float32)
    return P, Q


def run_fwd(P, Q):
    loss, dp, ip, dq, iq = ops.chamfer_fwd(dev(P), dev(Q))
    assert ops.device_status() == 0
    return (loss.cpu().numpy(), dp.cpu().numpy(), ip.cpu().numpy(), dq.cpu().numpy(), iq.cpu().numpy())


def sq64(X, Y, idx):
    """Exact squared distances (double) from every row of X to Y[idx]."""
    x = X.astype(np.float64)
    y = Y.astype(np.float64)[np.maximum(idx, 0)]
    return ((x - y) ** 2).sum(-1)


def search_error(dim):
    """Bound on |search value - exact| per unit of |x|^2 + |y|^2 (see above)."""
    return 2.0 ** -17 if dim <= 4 else 8 * U


def assert_nearest(X, Y, got, ref):
    """got: the kernel's nearest indices [n], ref: the oracle's [n] (one set)."""
    assert np.array_equal(got < 0, ref < 0)
    diff = got != ref
    if not diff.any():
        return
    x2 = (X.astype(np.float64) ** 2).sum(-1)
    y2 = (Y.astype(np.float64) ** 2).sum(-1)
    dg, dr = sq64(X, Y, got), sq64(X, Y, ref)
    tol = search_error(X.shape[-1]) * (2 * x2 + y2[np.maximum(got, 0)] + y2[np.maximum(ref, 0)])
    bad = diff & (dg > dr + tol)
    assert not bad.any(), f"{bad.sum()} of {diff.sum()} differing nearest indices are not within the fp32 bound"


def check_fwd(P, Q, exact=False):
    loss, dp, ip, dq, iq = run_fwd(P, Q)
    rdp, rip, _, rdq, riq, _, rloss = oracle.chamfer_fwd(P, Q)
    B = P.shape[0]
    for b in range(B):
        if exact:
            assert np.array_equal(ip[b], rip[b]) and np.array_equal(iq[b], riq[b])
            assert np.array_equal(dp[b].astype(np.float64), rdp[b])
            assert np.array_equal(dq[b].astype(np.float64), rdq[b])
        else:
            assert_nearest(P[b], Q[b], ip[b], rip[b])
            assert_nearest(Q[b], P[b], iq[b], riq[b])
            # the reported distance is the fp32 distance to the reported index
            for X, Y, d, i in ((P[b], Q[b], dp[b], ip[b]), (Q[b], P[b], dq[b], iq[b])):
                ref = sq64(X, Y, i)
                ref[i < 0] = 0.0
                assert np.allclose(d, ref, rtol=8 * U * X.shape[-1], atol=1e-30)
    assert np.allclose(loss, rloss, rtol=1e-5, atol=1e-6)
    return loss, ip, iq


@pytest.mark.parametrize("B,N,M", [(1, 1, 1), (3, 1000, 5000), (2, 4097, 300), (1, 2049, 8193), (2, 33, 31)])
def test_integer_clouds_exact(B, N, M):
    # many exact ties: the lowest index must win, as in the oracle
    P, Q = clouds(B * 1000 + N, B, N, M, 3, integer=True)
    check_fwd(P, Q, exact=True)


@pytest.mark.parametrize("dim", [1, 2, 3, 4, 5, 8])
def test_gaussian_clouds_every_dim(dim):
    P, Q = clouds(dim, 2, 3001, 4500, dim)
    check_fwd(P, Q)


def test_spans_tiles_and_sources_ragged():
    # source blocks of 2048 (dim 3) and target spans of 4096 with ragged tails
    P, Q = clouds(7, 1, 2048 * 2 + 5, 4096 * 2 + 33, 3)
    check_fwd(P, Q)


def test_empty_sets():
    P, Q = clouds(9, 2, 100, 0, 3)
    loss, dp, ip, dq, iq = run_fwd(P, Q)
    assert (loss == 0).all() and (ip == -1).all() and (dp == 0).all() and iq.size == 0
    loss, dp, ip, dq, iq = run_fwd(Q, P)
    assert (loss == 0).all() and (iq == -1).all() and (dq == 0).all() and ip.size == 0
    g = np.ones(2, np.float32)
    dP, dQ = ops.chamfer_bwd(dev(P), dev(Q), dev(np.full((2, 100), -1, np.int32)), dev(np.zeros((2, 0), np.int32)),
                             dev(g))
    assert ops.device_status() == 0
    assert (dP.cpu() == 0).all()


def test_duplicate_points_and_identical_sets():
    # coordinates on a 1/8 grid: every search value is exact, distinct points
    # are at least 1/64 apart in squared distance
    P, _ = clouds(11, 1, 500, 1, 3)
    P = np.clip(np.round(P * 8) / 8, -4, 4).astype(np.float32)
    P = np.concatenate([P, P[:, ::-1]], axis=1)  # every point at least twice
    loss, dp, ip, dq, iq = run_fwd(P, P)
    assert loss[0] == 0 and (dp == 0).all() and (dq == 0).all()
    first = {tuple(p): i for i, p in reversed(list(enumerate(P[0].tolist())))}
    want = np.array([first[tuple(p)] for p in P[0].tolist()])
    assert np.array_equal(ip[0], want) and np.array_equal(iq[0], want)


def bwd(P, Q, ip, iq, g):
    dP, dQ = ops.chamfer_bwd(dev(P), dev(Q), dev(ip), dev(iq), dev(g))
    assert ops.device_status() == 0
    return dP.cpu().numpy(), dQ.cpu().numpy()


def test_backward_integer_exact():
    # integer points, power-of-two set sizes and gradients: every term exact
    P, Q = clouds(13, 2, 1024, 4096, 3, integer=True)
    _, ip, iq = check_fwd(P, Q, exact=True)
    g = np.array([0.5, -2.0], np.float32)
    dP, dQ = bwd(P, Q, ip, iq, g)
    rP, rQ = oracle.chamfer_bwd(P, Q, ip, iq, g)
    assert np.array_equal(dP.astype(np.float64), rP) and np.array_equal(dQ.astype(np.float64), rQ)


@pytest.mark.parametrize("dim", [3, 7])
def test_backward_gaussian(dim):
    P, Q = clouds(17 + dim, 3, 2500, 1777, dim)
    _, ip, iq = check_fwd(P, Q)
    g = np.array([1.0, -0.25, 3.5], np.float32)
    dP, dQ = bwd(P, Q, ip, iq, g)
    rP, rQ = oracle.chamfer_bwd(P, Q, ip, iq, g)
    for got, ref in ((dP, rP), (dQ, rQ)):
        scale = np.abs(ref).max()
        assert np.allclose(got, ref, rtol=1e-5, atol=1e-6 * scale)
        g64 = got.astype(np.float64)
        cos = (g64 * ref).sum() / (np.linalg.norm(g64) * np.linalg.norm(ref))
        assert cos > 1 - 1e-9  # the pages report a gradient cosine of 1.00000 against autograd


def test_backward_is_bitwise_reproducible_and_hubs():
    # one target is the nearest of every source: a long inverse row
    P, Q = clouds(19, 1, 3000, 50, 3)
    Q[0, 7] = 0.0
    P[0] *= 1e-3
    _, ip, iq = check_fwd(P, Q)
    assert (ip == 7).all()
    g = np.array([1.5], np.float32)
    a = bwd(P, Q, ip, iq, g)
    b = bwd(P, Q, ip, iq, g)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    rP, rQ = oracle.chamfer_bwd(P, Q, ip, iq, g)
    assert np.allclose(a[0], rP, rtol=1e-5, atol=1e-7) and np.allclose(a[1], rQ, rtol=1e-4, atol=1e-6)


def test_backward_matches_an_fp32_model_bit_for_bit():
    # the kernel's own fp32 operations, in ascending source order along every
    # inverse row: equal to the last bit only if the inverse index is stable
    # and the formula is the stated one
    P, Q = clouds(37, 2, 300, 220, 3)
    _, ip, iq = check_fwd(P, Q)
    g = np.array([0.3, -1.7], np.float32)
    dP, dQ = bwd(P, Q, ip, iq, g)
    f = np.float32
    for b in range(2):
        for X, Y, near, inv_src, got in ((P[b], Q[b], ip[b], iq[b], dP[b]), (Q[b], P[b], iq[b], ip[b], dQ[b])):
            wx = f(f(2) * g[b]) / f(len(X))
            wy = f(f(2) * g[b]) / f(len(Y))
            for x in range(len(X)):
                inv = np.zeros(X.shape[1], np.float32)
                for y in np.nonzero(inv_src == x)[0]:  # ascending
                    inv = inv + (Y[y] - X[x])
                own = wx * (X[x] - Y[near[x]])
                assert np.array_equal(got[x], own - wy * inv), (b, x)


def test_backward_bad_index_is_reported_and_skipped():
    P, Q = clouds(23, 1, 200, 300, 3)
    _, ip, iq = check_fwd(P, Q)
    g = np.array([1.0], np.float32)
    bad = ip.copy()
    bad[0, 5] = 300 + 9
    dP, dQ = ops.chamfer_bwd(dev(P), dev(Q), dev(bad), dev(iq), dev(g))
    assert ops.device_status() == 6
    skip = ip.copy()
    skip[0, 5] = -1
    rP, rQ = oracle.chamfer_bwd(P, Q, skip, iq, g)
    assert np.allclose(dP.cpu().numpy(), rP, rtol=1e-5, atol=1e-7)
    assert np.allclose(dQ.cpu().numpy(), rQ, rtol=1e-5, atol=1e-7)


def test_autograd_matches_the_entry_points():
    P, Q = clouds(29, 2, 700, 900, 3)
    Pt = dev(P).requires_grad_(True)
    Qt = dev(Q).requires_grad_(True)
    loss = chamfer_distance(Pt, Qt)
    w = torch.tensor([0.75, -1.25], device="cuda")
    (loss * w).sum().backward()
    _, ip, iq = check_fwd(P, Q)
    rP, rQ = oracle.chamfer_bwd(P, Q, ip, iq, w.cpu().numpy())
    assert np.allclose(Pt.grad.cpu().numpy(), rP, rtol=1e-5, atol=1e-7)
    assert np.allclose(Qt.grad.cpu().numpy(), rQ, rtol=1e-5, atol=1e-7)


def test_full_size_clouds_sampled():
    # 100,000 x 100,000 points: the nearest index of 1,500 sampled points of
    # each cloud against the oracle, the loss from exact distances of every
    # reported index, and the whole backward against the oracle's
    w = workloads.make("chamfer_100k")
    P, Q, g = w["P"], w["Q"], w["grad"]
    loss, dp, ip, dq, iq = run_fwd(P, Q)
    rng = np.random.default_rng(31)
    for X, Y, idx in ((P, Q, ip), (Q, P, iq)):
        pick = np.sort(rng.choice(X.shape[1], size=1500, replace=False))
        _, ref_i, _, _, _, _, _ = oracle.chamfer_fwd(X[:, pick], Y)
        assert_nearest(X[0, pick], Y[0], idx[0, pick], ref_i[0])
    exact = sq64(P[0], Q[0], ip[0]).sum() / P.shape[1] + sq64(Q[0], P[0], iq[0]).sum() / Q.shape[1]
    assert abs(loss[0] - exact) <= 1e-5 * exact
    dP, dQ = bwd(P, Q, ip, iq, g)
    rP, rQ = oracle.chamfer_bwd(P, Q, ip, iq, g)
    for got, ref in ((dP, rP), (dQ, rQ)):
        assert np.allclose(got, ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())
