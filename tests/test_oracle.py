"""Pins for the CPU oracle: hand-worked values, an independent brute force,
closed forms, invariants and finite differences (no GPU)."""
import numpy as np
import pytest

import datagen
import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


# ---------------------------------------------------------------- hand-worked values

def test_hand_two_by_three(golden):
    ex = golden["two_by_three"]
    Q, D = f64(ex["Q"]), f64(ex["D"])
    for case in ex["cases"]:
        qm = None if case["q_mask"] is None else np.array(case["q_mask"], dtype=np.uint8)
        dm = None if case["d_mask"] is None else np.array(case["d_mask"], dtype=np.uint8)
        for dtype in ("f64", "f16", "bf16"):
            Qx = Q if dtype == "f64" else datagen.float_to_bits(Q, dtype)
            Dx = D if dtype == "f64" else datagen.float_to_bits(D, dtype)
            s, a, _ = oracle.fwd_dense(Qx, Dx, dtype, q_mask=qm, d_mask=dm)
            assert s[0, 0] == case["score"], (case["name"], dtype)
            assert a[0].tolist() == case["argmax"], (case["name"], dtype)


def test_hand_backward(golden):
    ex = golden["two_by_three"]
    Q, D = f64(ex["Q"]), f64(ex["D"])
    _, a, _ = oracle.fwd_dense(Q, D, "f64")
    dQ, dD, rp, col = oracle.bwd(Q, D, "f64", a, np.ones((1, 1), np.float32))
    bw = ex["backward_g1"]
    assert np.array_equal(dQ, f64(bw["dQ"]))
    assert np.array_equal(dD, f64(bw["dD"]))
    assert rp.tolist() == bw["row_ptr"]
    assert col.tolist() == bw["col"]


def test_negative_scores_masked_before_max(golden):
    ex = golden["negative_scores"]
    Q, D = f64(ex["Q"]), f64(ex["D"])
    for case in ex["cases"]:
        dm = None if case["d_mask"] is None else np.array(case["d_mask"], dtype=np.uint8)
        s, a, _ = oracle.fwd_dense(Q, D, "f64", d_mask=dm)
        assert s[0, 0] == case["score"]
        assert a[0].tolist() == case["argmax"]


def test_tie_lowest_index(golden):
    ex = golden["tie"]
    s, a, g = oracle.fwd_dense(f64(ex["Q"]), f64(ex["D"]), "f64")
    assert s[0, 0] == ex["score"] and a[0].tolist() == ex["argmax"] and g[0].tolist() == ex["gap"]


def test_all_masked_doc_sentinel(golden):
    ex = golden["all_masked_doc"]
    s, a, g = oracle.fwd_dense(f64(ex["Q"]), f64(ex["D"]), "f64", d_mask=np.array(ex["d_mask"], np.uint8))
    assert s[0, 0] == ex["score"] and a[0].tolist() == ex["argmax"]
    assert np.all(np.isinf(g))
    # the backward routes nothing through a sentinel
    dQ, dD, rp, col = oracle.bwd(f64(ex["Q"]), f64(ex["D"]), "f64", a, np.ones((1, 1), np.float32))
    assert not dQ.any() and not dD.any() and rp[-1] == 0 and col.size == 0


def test_int8_scale_flip(golden):
    ex = golden["int8_scale_flip"]
    Q = np.array(ex["Q"], np.int8)
    D = np.array(ex["D"], np.int8)
    s, a, w, _ = oracle.fwd_int8(Q, np.array(ex["q_scale"], np.float32), D, np.array(ex["d_scale"], np.float32))
    assert abs(s[0, 0] - ex["score"]) < 1e-12  # 0.1 is not exact in binary
    assert a[0].tolist() == ex["argmax"] and w[0].tolist() == ex["win_dot"]


# ---------------------------------------------------------------- decoders

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decoder_matches_numpy_on_all_finite_patterns(dtype):
    # Every finite bit pattern, decoded by the oracle (via a 1x1 product with 1.0)
    # must equal numpy's own conversion of the same bits.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = datagen.bits_to_float(bits, dtype)
    keep = np.isfinite(vals)
    bits, vals = bits[keep], vals[keep]
    n = bits.size
    Q = bits.reshape(n, 1, 1).copy()
    one = datagen.float_to_bits(np.ones((1, 1, 1)), dtype)
    s, _, _ = oracle.fwd_dense(Q, one, dtype)
    assert np.array_equal(s[:, 0], vals)


# ---------------------------------------------------------------- brute force

def brute_force(Qf, Df, q_mask=None, d_mask=None):
    """Independent einsum-then-reduce restatement: materialise S, mask, max, sum."""
    S = np.einsum("isk,jtk->ijst", Qf, Df)  # [Nq, Nd, Lq, Ld]
    if d_mask is not None:
        S = np.where(d_mask[None, :, None, :].astype(bool), S, -np.inf)
    m = S.max(axis=3) if S.shape[3] else np.full(S.shape[:3], -np.inf)
    arg = np.where(np.isfinite(m), S.argmax(axis=3) if S.shape[3] else 0, -1)
    active = np.ones(Qf.shape[:2], bool) if q_mask is None else q_mask.astype(bool)
    contrib = np.where(np.isfinite(m) & active[:, None, :], m, 0.0)
    return contrib.sum(axis=2), arg.reshape(-1, Qf.shape[1])


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_brute_force_tiny(seed, dtype):
    rng = np.random.default_rng(seed)
    Nq, Nd = rng.integers(1, 4, size=2)
    Lq, Ld = rng.integers(1, 8, size=2)
    dim = int(rng.integers(1, 9))
    Q = datagen.gaussian_rows(100 + seed, 1, Nq * Lq, dim, dtype).reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(100 + seed, 2, Nd * Ld, dim, dtype).reshape(Nd, Ld, dim)
    qm = (rng.random((Nq, Lq)) > 0.3).astype(np.uint8)
    dm = (rng.random((Nd, Ld)) > 0.3).astype(np.uint8)
    Qf, Df = datagen.bits_to_float(Q, dtype), datagen.bits_to_float(D, dtype)
    for q_mask, d_mask in ((None, None), (qm, None), (None, dm), (qm, dm)):
        s, a, g = oracle.fwd_dense(Q, D, dtype, q_mask=q_mask, d_mask=d_mask)
        bs, ba = brute_force(Qf, Df, q_mask, d_mask)
        np.testing.assert_allclose(s, bs, rtol=1e-12, atol=1e-12)
        clear = g > 1e-9
        assert np.array_equal(a[clear], ba[clear])
        assert np.array_equal(a == -1, ba == -1)


def test_top2_gap_is_max_minus_second():
    rng = np.random.default_rng(7)
    Q = f64(rng.standard_normal((2, 3, 4)))
    D = f64(rng.standard_normal((3, 5, 4)))
    _, _, g = oracle.fwd_dense(Q, D, "f64")
    S = np.einsum("isk,jtk->ijst", Q, D)
    top = np.sort(S, axis=3)
    np.testing.assert_allclose(g.reshape(2, 3, 3), top[..., -1] - top[..., -2], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_single_doc_token_closed_form():
    rng = np.random.default_rng(1)
    Q = f64(rng.standard_normal((3, 6, 8)))
    D = f64(rng.standard_normal((4, 1, 8)))
    s, a, _ = oracle.fwd_dense(Q, D, "f64")
    np.testing.assert_allclose(s, Q.sum(axis=1) @ D[:, 0, :].T, rtol=1e-12, atol=1e-12)
    assert (a == 0).all()


def test_single_query_token_closed_form():
    rng = np.random.default_rng(2)
    Q = f64(rng.standard_normal((1, 1, 16)))
    D = f64(rng.standard_normal((5, 9, 16)))
    s, a, _ = oracle.fwd_dense(Q, D, "f64")
    mv = D @ Q[0, 0]  # [Nd, Ld] textbook mat-vec
    np.testing.assert_allclose(s[0], mv.max(axis=1), rtol=1e-12, atol=1e-12)
    assert np.array_equal(a[:, 0], mv.argmax(axis=1))


def test_positive_homogeneity():
    rng = np.random.default_rng(3)
    Q = f64(rng.standard_normal((2, 4, 8)))
    D = f64(rng.standard_normal((3, 7, 8)))
    s1, a1, _ = oracle.fwd_dense(Q, D, "f64")
    s2, a2, _ = oracle.fwd_dense(f64(2.0 * Q), D, "f64")
    assert np.array_equal(s2, 2.0 * s1) and np.array_equal(a1, a2)


# ---------------------------------------------------------------- invariants

def test_chunking_identity():
    # Splitting Q into 128-token chunks and summing the chunk scores equals the
    # full score (design notes, "Long-query chunking").
    Nq, Lq, Nd, Ld, dim = 2, 1024, 3, 40, 16
    Q = datagen.gaussian_rows(5, 1, Nq * Lq, dim, "bf16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(5, 2, Nd * Ld, dim, "bf16").reshape(Nd, Ld, dim)
    qm = datagen.mask_drop_tail(5, 4, Nq, Lq, 300)
    full, a_full, _ = oracle.fwd_dense(Q, D, "bf16", q_mask=qm)
    nc = Lq // 128
    sc, a_c, _ = oracle.fwd_dense(Q.reshape(Nq * nc, 128, dim), D, "bf16", q_mask=qm.reshape(Nq * nc, 128))
    np.testing.assert_allclose(sc.reshape(Nq, nc, Nd).sum(axis=1), full, rtol=0, atol=1e-12)
    # argmax in original token layout
    a_c = a_c.reshape(Nq, nc, Nd, 128).transpose(0, 2, 1, 3).reshape(Nq * Nd, Lq)
    assert np.array_equal(a_c, a_full)


def test_mask_invariants():
    Nq, Lq, Nd, Ld, dim = 3, 9, 4, 13, 8
    Q = datagen.gaussian_rows(9, 1, Nq * Lq, dim, "f16").reshape(Nq, Lq, dim)
    D = datagen.gaussian_rows(9, 2, Nd * Ld, dim, "f16").reshape(Nd, Ld, dim)
    base, a0, _ = oracle.fwd_dense(Q, D, "f16")
    ones_s, ones_a, _ = oracle.fwd_dense(Q, D, "f16", q_mask=np.ones((Nq, Lq), np.uint8),
                                         d_mask=np.ones((Nd, Ld), np.uint8))
    assert np.array_equal(base, ones_s) and np.array_equal(a0, ones_a)
    # trailing d_mask of k tokens == varlen documents of length Ld - k
    k = np.array([0, 3, Ld, 5])
    dm = np.ones((Nd, Ld), np.uint8)
    for j in range(Nd):
        dm[j, Ld - k[j]:] = 0
    ms, ma, _ = oracle.fwd_dense(Q, D, "f16", d_mask=dm)
    lens = Ld - k
    rows = np.concatenate([D[j, :lens[j]] for j in range(Nd)]).reshape(-1, dim)
    d_off = np.concatenate([[0], np.cumsum(lens)])
    q_off = np.arange(Nq + 1) * Lq
    vs, va, _ = oracle.fwd_packed(Q.reshape(-1, dim), q_off, rows, d_off, "f16")
    assert np.array_equal(ms, vs) and np.array_equal(ma, va)
    assert (vs[:, 2] == 0).all() and (va.reshape(Nq, Nd, Lq)[:, 2] == -1).all()  # empty doc
    # q_mask = 0 on a row == deleting the row
    qm = np.ones((Nq, Lq), np.uint8)
    qm[:, 4] = 0
    s_masked, _, _ = oracle.fwd_dense(Q, D, "f16", q_mask=qm)
    s_del, _, _ = oracle.fwd_dense(np.ascontiguousarray(np.delete(Q, 4, axis=1)), D, "f16")
    assert np.array_equal(s_masked, s_del)
    # permuting document tokens permutes the argmax and keeps the score
    perm = np.random.default_rng(0).permutation(Ld)
    ps, pa, pg = oracle.fwd_dense(Q, np.ascontiguousarray(D[:, perm]), "f16")
    np.testing.assert_allclose(ps, base, rtol=0, atol=1e-12)
    clear = pg > 0
    assert np.array_equal(perm[pa[clear]], a0[clear])


def _ragged_problem(seed, lq_lens, ld_lens, dim, dtype):
    """Packed queries / documents of the given lengths with random masks (one
    byte per packed row)."""
    rng = np.random.default_rng(seed)
    q_off = np.concatenate([[0], np.cumsum(lq_lens)]).astype(np.int64)
    d_off = np.concatenate([[0], np.cumsum(ld_lens)]).astype(np.int64)
    Q = datagen.gaussian_rows(300 + seed, 1, int(q_off[-1]), dim, dtype)
    D = datagen.gaussian_rows(300 + seed, 2, int(d_off[-1]), dim, dtype)
    qm = (rng.random(int(q_off[-1])) > 0.3).astype(np.uint8)
    dm = (rng.random(int(d_off[-1])) > 0.3).astype(np.uint8)
    return Q, q_off, D, d_off, qm, dm


def test_packed_queries_equal_padded_dense():
    # Packed queries of lengths L_i ("late-interaction-kernels" notes, "Varlen /
    # packed path": cu_seqlens on both sides) score exactly like dense queries
    # padded to max L_i whose padding rows carry q_mask = 0 (the notes' "Problem":
    # q_mask drops a row from the sum). Rows past a query's end report -1.
    dim, dtype = 8, "bf16"
    lq_lens = np.array([3, 7, 1, 5])
    ld_lens = np.array([4, 0, 9, 2, 6])
    Q, q_off, D, d_off, qm, dm = _ragged_problem(41, lq_lens, ld_lens, dim, dtype)
    Nq, Nd, max_lq = len(lq_lens), len(ld_lens), int(lq_lens.max())
    for q_mask, d_mask in ((None, None), (qm, None), (None, dm), (qm, dm)):
        s, a, g = oracle.fwd_packed(Q, q_off, D, d_off, dtype, q_mask=q_mask, d_mask=d_mask)
        assert a.shape == (Nq * Nd, max_lq)
        # dense padded twin: padding rows hold unrelated values and q_mask = 0
        Qd = datagen.gaussian_rows(77, 1, Nq * max_lq, dim, dtype).reshape(Nq, max_lq, dim)
        qmd = np.zeros((Nq, max_lq), np.uint8)
        for i in range(Nq):
            L = lq_lens[i]
            Qd[i, :L] = Q[q_off[i]:q_off[i + 1]]
            qmd[i, :L] = 1 if q_mask is None else q_mask[q_off[i]:q_off[i + 1]]
        ds_, da, _ = oracle.fwd_packed(Qd.reshape(-1, dim), np.arange(Nq + 1) * max_lq, D, d_off, dtype,
                                       q_mask=qmd.reshape(-1), d_mask=d_mask)
        assert np.array_equal(s, ds_)
        for i in range(Nq):
            L = lq_lens[i]
            rows = slice(i * Nd, (i + 1) * Nd)
            assert np.array_equal(a[rows, :L], da[rows, :L])
            assert (a[rows, L:] == -1).all() and np.isinf(g[rows, L:]).all()


@pytest.mark.parametrize("seed", range(4))
def test_packed_queries_brute_force(seed):
    # Independent per-pair restatement on ragged queries and documents: slice the
    # query's and the document's rows by their offsets, form S, hide masked
    # document rows with -inf, take the row maxima and sum over active rows.
    rng = np.random.default_rng(500 + seed)
    dim = int(rng.integers(1, 9))
    lq_lens = rng.integers(0, 7, size=int(rng.integers(1, 5)))
    ld_lens = rng.integers(0, 8, size=int(rng.integers(1, 5)))
    Q, q_off, D, d_off, qm, dm = _ragged_problem(seed, lq_lens, ld_lens, dim, "f16")
    Qf, Df = datagen.bits_to_float(Q, "f16"), datagen.bits_to_float(D, "f16")
    Nq, Nd = len(lq_lens), len(ld_lens)
    s, a, g = oracle.fwd_packed(Q, q_off, D, d_off, "f16", q_mask=qm, d_mask=dm)
    for i in range(Nq):
        qi = Qf[q_off[i]:q_off[i + 1]]
        act = qm[q_off[i]:q_off[i + 1]].astype(bool)
        for j in range(Nd):
            S = qi @ Df[d_off[j]:d_off[j + 1]].T  # [L_i, Ld_j]
            S = np.where(dm[d_off[j]:d_off[j + 1]].astype(bool)[None, :], S, -np.inf)
            m = S.max(axis=1) if S.shape[1] else np.full(S.shape[0], -np.inf)
            want = np.where(np.isfinite(m) & act, m, 0.0).sum()
            assert abs(s[i, j] - want) <= 1e-12 * max(1.0, abs(want))
            arg = np.where(np.isfinite(m), S.argmax(axis=1) if S.shape[1] else 0, -1)
            row = a[i * Nd + j, : len(m)]
            clear = g[i * Nd + j, : len(m)] > 1e-9
            assert np.array_equal(row[clear], arg[clear]) and np.array_equal(row == -1, arg == -1)


# ---------------------------------------------------------------- INT8

def test_int8_brute_force():
    Nq, Lq, Nd, Ld, dim = 2, 5, 3, 11, 32
    q, qs = datagen.int8_rows(11, 1, Nq * Lq, dim)
    d, ds = datagen.int8_rows(11, 2, Nd * Ld, dim)
    dm = (np.random.default_rng(3).random((Nd, Ld)) > 0.2).astype(np.uint8)
    Q, D = q.reshape(Nq, Lq, dim), d.reshape(Nd, Ld, dim)
    s, a, w, _ = oracle.fwd_int8(Q, qs.reshape(Nq, Lq), D, ds.reshape(Nd, Ld), d_mask=dm)
    dots = np.einsum("isk,jtk->ijst", Q.astype(np.int64), D.astype(np.int64))
    v = dots * ds.reshape(Nd, Ld).astype(np.float64)[None, :, None, :]
    v = np.where(dm[None, :, None, :].astype(bool), v, -np.inf)
    am = v.argmax(axis=3)
    want = (v.max(axis=3) * qs.reshape(Nq, Lq).astype(np.float64)[:, None, :]).sum(axis=2)
    np.testing.assert_allclose(s, want, rtol=1e-12)
    assert np.array_equal(a.reshape(Nq, Nd, Lq), am)
    assert np.array_equal(w.reshape(Nq, Nd, Lq), np.take_along_axis(dots, am[..., None], axis=3)[..., 0])


def test_int8_quantisation_recipe():
    q, s = datagen.int8_rows(1, 2, 64, 128)
    x = datagen.gaussian_rows(1, 2, 64, 128, "f64")
    assert (np.abs(q).max(axis=1) == 127).all()  # the largest entry maps to +-127
    np.testing.assert_allclose(s, (np.abs(x).max(axis=1) / 127).astype(np.float32), rtol=0)
    assert (np.abs(q.astype(np.float64) * s[:, None] - x) <= s[:, None] * 0.5 + 1e-12).all()


# ---------------------------------------------------------------- backward

def small_problem(seed=21, Nq=3, Lq=6, Nd=4, Ld=9, dim=8):
    rng = np.random.default_rng(seed)
    Q = f64(rng.standard_normal((Nq, Lq, dim)))
    D = f64(rng.standard_normal((Nd, Ld, dim)))
    g = rng.standard_normal((Nq, Nd)).astype(np.float32)
    qm = (rng.random((Nq, Lq)) > 0.25).astype(np.uint8)
    return Q, D, g, qm


def test_backward_euler_identity():
    # score is positively 1-homogeneous in Q and in D, so
    # sum <dQ, Q> = sum g * score = sum <dD, D>.
    Q, D, g, qm = small_problem()
    s, a, _ = oracle.fwd_dense(Q, D, "f64", q_mask=qm)
    dQ, dD, _, _ = oracle.bwd(Q, D, "f64", a, g, q_mask=qm)
    target = float((g.astype(np.float64) * s).sum())
    assert abs((dQ * Q).sum() - target) < 1e-10
    assert abs((dD * D).sum() - target) < 1e-10


def test_backward_finite_differences():
    Q, D, g, qm = small_problem(seed=5, Nq=2, Lq=4, Nd=3, Ld=5, dim=4)
    s, a, gap = oracle.fwd_dense(Q, D, "f64", q_mask=qm)
    assert gap.min() > 1e-3  # differentiable point for this seed
    dQ, dD, _, _ = oracle.bwd(Q, D, "f64", a, g, q_mask=qm)
    gd = g.astype(np.float64)

    def loss(Qx, Dx):
        return float((gd * oracle.fwd_dense(f64(Qx), f64(Dx), "f64", q_mask=qm)[0]).sum())

    h = 1e-6
    for idx in np.ndindex(Q.shape):
        Qp, Qn = Q.copy(), Q.copy()
        Qp[idx] += h
        Qn[idx] -= h
        assert abs((loss(Qp, D) - loss(Qn, D)) / (2 * h) - dQ[idx]) < 1e-6
    for idx in np.ndindex(D.shape):
        Dp, Dn = D.copy(), D.copy()
        Dp[idx] += h
        Dn[idx] -= h
        assert abs((loss(Q, Dp) - loss(Q, Dn)) / (2 * h) - dD[idx]) < 1e-6


def test_backward_column_sums_and_csr():
    Q, D, g, qm = small_problem(seed=8, Nq=4, Lq=5, Nd=3, Ld=6)
    dm = np.ones((3, 6), np.uint8)
    dm[1] = 0  # a fully masked document produces sentinels
    s, a, _ = oracle.fwd_dense(Q, D, "f64", q_mask=qm, d_mask=dm)
    dQ, dD, rp, col = oracle.bwd(Q, D, "f64", a, g, q_mask=qm)
    Nq, Lq, Nd, Ld = 4, 5, 3, 6
    # sum_t dD[j,t] = sum_i g_ij sum_s q_mask * Q[i,s]  (for documents with a winner)
    qsum = (Q * qm[..., None]).sum(axis=1)
    want = g.astype(np.float64).T @ qsum
    want[1] = 0
    np.testing.assert_allclose(dD.sum(axis=1), want, rtol=1e-12, atol=1e-12)
    # CSR: row_ptr is the exclusive scan of a direct histogram; sources ascend
    src = np.arange(Nq * Nd * Lq)
    av = a.reshape(-1)
    keep = av >= 0
    dest = ((src // Lq) % Nd) * Ld + av
    hist = np.bincount(dest[keep], minlength=Nd * Ld)
    assert np.array_equal(np.diff(rp), hist) and rp[0] == 0 and rp[-1] == keep.sum()
    assert np.array_equal(col, np.argsort(np.where(keep, dest, Nd * Ld), kind="stable")[: keep.sum()])
    # dQ gathers exactly one D row per document
    i, s_ = 2, 3
    w = qm[i, s_]
    want_q = sum(g[i, j] * D[j, a[i * Nd + j, s_]] for j in range(Nd) if a[i * Nd + j, s_] >= 0) * w
    np.testing.assert_allclose(dQ[i, s_], want_q, rtol=1e-12, atol=1e-12)


def test_csr_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.csr(np.array([[0, 7]], np.int32), 1, 2, 1, 3)


# ---------------------------------------------------------------- Chamfer distance

def test_chamfer_hand_example(golden):
    ex = golden["chamfer_two_points"]
    P = np.array([ex["P"]], np.float32)
    Q = np.array([ex["Q"]], np.float32)
    dp, ip, _, dq, iq, _, loss = oracle.chamfer_fwd(P, Q)
    assert dp[0].tolist() == ex["dist_p"] and ip[0].tolist() == ex["idx_p"]
    assert dq[0].tolist() == ex["dist_q"] and iq[0].tolist() == ex["idx_q"]
    assert loss[0] == ex["loss"]
    dP, dQ = oracle.chamfer_bwd(P, Q, ip, iq, np.array([ex["grad_loss"]], np.float32))
    assert dP[0].tolist() == ex["dP"] and dQ[0].tolist() == ex["dQ"]


def _clouds(seed, B, N, M, dim=3, scale=1.0, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        return (rng.integers(-20, 21, (B, N, dim)).astype(np.float32), rng.integers(-20, 21, (B, M, dim)).astype(np.float32))
    return ((rng.standard_normal((B, N, dim)) * scale).astype(np.float32),
            (rng.standard_normal((B, M, dim)) * scale).astype(np.float32))


def _sq_dist(p, q):
    """Squared distance summed left to right in double (the built-in sum() of
    floats compensates, which would round differently)."""
    d = 0.0
    for x, y in zip(p, q):
        t = float(x) - float(y)
        d += t * t
    return d


def test_chamfer_brute_force_tiny():
    # nearest neighbours by exhaustive search over an explicit distance table
    for seed in range(5):
        P, Q = _clouds(seed, 2, 7, 5, dim=1 + seed % 4)
        dp, ip, gp, dq, iq, gq, loss = oracle.chamfer_fwd(P, Q)
        for b in range(2):
            table = np.array([[_sq_dist(p, q) for q in Q[b]] for p in P[b]])
            assert np.array_equal(ip[b], table.argmin(axis=1)) and np.array_equal(iq[b], table.argmin(axis=0))
            assert np.array_equal(dp[b], table.min(axis=1)) and np.array_equal(dq[b], table.min(axis=0))
            assert np.array_equal(gp[b], np.sort(table, axis=1)[:, 1] - table.min(axis=1))
            # sums in a different order: equal to rounding
            assert np.isclose(loss[b], table.min(axis=1).mean() + table.min(axis=0).mean(), rtol=1e-14, atol=0)


def test_chamfer_invariants():
    P, Q = _clouds(11, 3, 40, 33, integer=True)
    _, _, _, _, _, _, loss = oracle.chamfer_fwd(P, Q)
    # symmetric in its arguments
    assert np.array_equal(oracle.chamfer_fwd(Q, P)[6], loss)
    # translation invariant (integer shifts keep every value exact)
    t = np.array([3, -7, 11], np.float32)
    assert np.array_equal(oracle.chamfer_fwd(P + t, Q + t)[6], loss)
    # a set against itself: zero, every point its own nearest neighbour
    dp, ip, _, dq, iq, _, l0 = oracle.chamfer_fwd(P, P)
    assert (l0 == 0).all() and (dp == 0).all() and (dq == 0).all()
    # scaling by 2 scales every squared distance by 4
    assert np.array_equal(oracle.chamfer_fwd(2 * P, 2 * Q)[6], 4 * loss)


def test_chamfer_single_target_closed_form():
    P, Q = _clouds(13, 2, 9, 1)
    dp, ip, _, dq, iq, _, loss = oracle.chamfer_fwd(P, Q)
    d = ((P.astype(np.float64) - Q.astype(np.float64)) ** 2).sum(-1)
    assert np.allclose(dp, d, rtol=1e-15, atol=0) and (ip == 0).all()
    assert np.allclose(dq[:, 0], d.min(axis=1), rtol=1e-15, atol=0)
    assert np.allclose(loss, d.mean(axis=1) + d.min(axis=1), rtol=1e-14, atol=0)


def test_chamfer_ties_take_lowest_index_and_empty_sets():
    P = np.zeros((1, 3, 3), np.float32)
    Q = np.array([[[1, 0, 0], [0, 1, 0], [0, 0, 1]]], np.float32)
    dp, ip, gp, dq, iq, _, _ = oracle.chamfer_fwd(P, Q)
    assert (ip == 0).all() and (gp == 0).all() and (iq == 0).all()
    dp, ip, _, dq, iq, _, loss = oracle.chamfer_fwd(np.zeros((1, 0, 3), np.float32), Q)
    assert loss[0] == 0 and (iq == -1).all() and (dq == 0).all()
    dP, dQ = oracle.chamfer_bwd(np.zeros((1, 0, 3), np.float32), Q, ip, iq, np.ones(1, np.float32))
    assert (dQ == 0).all()


def test_chamfer_gradient_finite_differences():
    P, Q = _clouds(17, 1, 12, 10)
    _, ip, gp, _, iq, gq, _ = oracle.chamfer_fwd(P, Q)
    assert gp.min() > 1e-3 and gq.min() > 1e-3  # nearest neighbours stable under the probe
    g = np.array([0.7], np.float32)
    dP, dQ = oracle.chamfer_bwd(P, Q, ip, iq, g)
    h = 1e-3

    def loss_at(P2, Q2):  # the loss at perturbed points, evaluated in double through the oracle's indices
        Pd, Qd = P2.astype(np.float64)[0], Q2.astype(np.float64)[0]
        return 0.7 * (((Pd - Qd[ip[0]]) ** 2).sum(-1).mean() + ((Qd - Pd[iq[0]]) ** 2).sum(-1).mean())

    for which, X, dX in (("P", P, dP), ("Q", Q, dQ)):
        for n, k in [(0, 0), (3, 1), (7, 2)]:
            Xp, Xm = X.astype(np.float64).copy(), X.astype(np.float64).copy()
            Xp[0, n, k] += h
            Xm[0, n, k] -= h
            if which == "P":
                fd = (loss_at(Xp, Q) - loss_at(Xm, Q)) / (2 * h)
            else:
                fd = (loss_at(P, Xp) - loss_at(P, Xm)) / (2 * h)
            assert abs(fd - dX[0, n, k]) < 1e-6 * max(1.0, abs(fd))


def test_chamfer_gradient_sums():
    # translation invariance of the loss: every gradient sums to zero over both sets
    P, Q = _clouds(19, 2, 30, 25)
    _, ip, _, _, iq, _, _ = oracle.chamfer_fwd(P, Q)
    dP, dQ = oracle.chamfer_bwd(P, Q, ip, iq, np.array([1.3, -0.4], np.float32))
    assert np.allclose(dP.sum(axis=1) + dQ.sum(axis=1), 0, atol=1e-12)


# ---------------------------------------------------------------- top-k and the two-stage scan

def _f16_bits(x):
    return datagen.float_to_bits(np.asarray(x, dtype=np.float64), "f16")


def test_two_stage_hand_example(golden):
    ex = golden["two_stage_topk"]
    Q8 = np.array(ex["Q8"], np.int8)
    D8 = np.array(ex["D8"], np.int8)
    qs = np.array(ex["q_scale"], np.float32)
    ds = np.array(ex["d_scale"], np.float32)
    Q16, D16 = _f16_bits(ex["Q16"]), _f16_bits(ex["D16"])
    top_idx, top_scores, s8, cand, s16 = oracle.two_stage_topk(Q8, qs, D8, ds, Q16, D16, "f16", ex["k1"], ex["k"])
    assert s8.tolist() == ex["s8"] and cand.tolist() == ex["candidates"] and s16.tolist() == ex["s16"]
    assert top_idx.tolist() == ex["top_idx"] and top_scores.tolist() == ex["top_scores"]


def test_topk_brute_force_with_ties_and_signed_zeros():
    rng = np.random.default_rng(71)
    for trial in range(20):
        n = int(rng.integers(1, 60))
        v = rng.integers(-4, 5, size=(3, n)).astype(np.float64) * 0.5
        v[:, ::7] = -0.0
        v[:, 1::9] = 0.0
        k = int(rng.integers(1, n + 1))
        idx, vals = oracle.topk(v, k)
        for r in range(3):
            want = sorted(range(n), key=lambda j: (-v[r, j], j))[:k]
            assert idx[r].tolist() == want
            assert vals[r].tolist() == [v[r, j] for j in want]
    # k = n: a permutation, descending
    v = rng.standard_normal((2, 50))
    idx, vals = oracle.topk(v, 50)
    assert all(sorted(row) == list(range(50)) for row in idx.tolist()) and (np.diff(vals, axis=1) <= 0).all()


def _two_stage_inputs(seed, Nq, Lq, Nd, Ld, dim, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        q = rng.integers(-3, 4, size=(Nq, Lq, dim))
        d = rng.integers(-3, 4, size=(Nd, Ld, dim))
        Q8, D8 = q.astype(np.int8), d.astype(np.int8)
        qs, ds = np.ones((Nq, Lq), np.float32), np.ones((Nd, Ld), np.float32)
        return Q8, qs, D8, ds, _f16_bits(q), _f16_bits(d)
    Q8, qs = datagen.int8_rows(seed, datagen.TID_Q, Nq * Lq, dim)
    D8, ds = datagen.int8_rows(seed, datagen.TID_D, Nd * Ld, dim)
    Q16 = datagen.gaussian_rows(seed, datagen.TID_Q, Nq * Lq, dim, "f16")
    D16 = datagen.gaussian_rows(seed, datagen.TID_D, Nd * Ld, dim, "f16")
    return (Q8.reshape(Nq, Lq, dim), qs.reshape(Nq, Lq), D8.reshape(Nd, Ld, dim), ds.reshape(Nd, Ld),
            Q16.reshape(Nq, Lq, dim), D16.reshape(Nd, Ld, dim))


def test_two_stage_with_every_candidate_is_the_exact_topk():
    Q8, qs, D8, ds, Q16, D16 = _two_stage_inputs(73, 3, 5, 40, 7, 32)
    top_idx, top_scores, s8, cand, s16 = oracle.two_stage_topk(Q8, qs, D8, ds, Q16, D16, "f16", 40, 6)
    exact, _, _ = oracle.fwd_dense(Q16, D16, "f16")
    want_idx, want_scores = oracle.topk(exact, 6)
    assert np.array_equal(top_idx, want_idx) and np.array_equal(top_scores, want_scores)
    # the candidates are every document, ordered by the INT8 scores
    assert all(sorted(row) == list(range(40)) for row in cand.tolist())


def test_two_stage_properties_and_integer_agreement():
    # integer embeddings with unit scales: both stages compute the same exact scores
    Q8, qs, D8, ds, Q16, D16 = _two_stage_inputs(79, 2, 4, 60, 5, 32, integer=True)
    top_idx, top_scores, s8, cand, s16 = oracle.two_stage_topk(Q8, qs, D8, ds, Q16, D16, "f16", 20, 8)
    assert np.array_equal(s16, np.take_along_axis(s8, cand.astype(np.int64), axis=1))
    want_idx, want_scores = oracle.topk(s8, 8)
    assert np.array_equal(top_idx, want_idx) and np.array_equal(top_scores, want_scores)
    # Gaussian embeddings: the final documents are candidates, scores descending, and each
    # final score is the f16 score of its document
    Q8, qs, D8, ds, Q16, D16 = _two_stage_inputs(83, 2, 6, 50, 9, 32)
    top_idx, top_scores, s8, cand, s16 = oracle.two_stage_topk(Q8, qs, D8, ds, Q16, D16, "f16", 12, 5)
    exact, _, _ = oracle.fwd_dense(Q16, D16, "f16")
    for i in range(2):
        assert set(top_idx[i].tolist()) <= set(cand[i].tolist())
        assert (np.diff(top_scores[i]) <= 0).all()
        assert np.array_equal(top_scores[i], exact[i, top_idx[i]])
