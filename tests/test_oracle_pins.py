"""Pins of the CPU oracle to facts fixed outside itself.

Each check is a function of the oracle's outputs, so the same check is run
on planted mistakes (a dropped column, a transposed operand, a missing
scale) to show it would catch them.  Citations name sections/equations of
"PuzzleKV: Page-Wise Low-Rank Decomposition for KV Cache Compression".
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_printed_values.json")


def _page(P, d, seed, k=6, n_out=2):
    spec = synth.KVSpec(layers=1, kv_heads=1, head_dim=d, page_size=P, inner_rank=k,
                        n_outliers=n_out, dtype=torch.float32)
    K, _ = synth.prefill_kv(spec, P, seq=seed)
    return K[0, 0].double().numpy()


# ---------------------------------------------------------------- SVD pins

def eckart_young_defect(X, L, R, S, r):
    """| ||X - L R||_F^2 - sum_{i>r} S_i^2 | / ||X||_F^2  (§3.2: the rank-r
    truncation attains the discarded singular-value energy)."""
    err = np.sum((X - L @ R) ** 2)
    tail = np.sum(S[r:] ** 2)
    tot = np.sum(X ** 2)
    return max(abs(err - tail), abs(tot - np.sum(S ** 2))) / max(tot, 1e-300)


def orthonormality_defect(L, R, S, r):
    """max of |L^T L - I| and |R R^T - diag(S_r^2)| / S_1^2."""
    a = np.abs(L.T @ L - np.eye(r)).max()
    b = np.abs(R @ R.T - np.diag(S[:r] ** 2)).max() / max(S[0] ** 2, 1e-300)
    return max(a, b)


@pytest.mark.parametrize("P,d,r", [(4, 4, 1), (4, 4, 2), (16, 32, 5), (32, 64, 8), (32, 64, 32), (64, 128, 16), (64, 128, 24)])
def test_eckart_young_and_orthonormality(P, d, r):
    for seed in range(3):
        X = _page(P, d, seed, k=min(6, P))
        L, R, S = oracle.factorize(X, r)
        assert eckart_young_defect(X, L, R, S, r) < 1e-12
        assert orthonormality_defect(L, R, S, r) < 1e-12
        assert np.all(np.diff(S) <= 0)


def test_singular_values_match_lapack():
    rng = np.random.default_rng(1)
    for P, d in [(4, 4), (8, 8), (32, 64), (64, 128)]:
        X = rng.standard_normal((P, d)) * rng.uniform(0.1, 10, size=(1, d))
        _, S, _, sweeps = oracle.svd(X)
        ref = np.linalg.svd(X, compute_uv=False)
        assert sweeps > 0
        assert np.abs(S - ref).max() <= 1e-12 * ref[0]


def test_gram_route_gives_the_same_factors():
    """PuzzleKV §3.3: the top-r eigenvectors Q_r of the Gram matrix X X^T give
    L = Q_r and R = Q_r^T X, the same rank-r factorization as the truncated
    SVD.  The oracle's one-sided Jacobi on X must match LAPACK's symmetric
    eigensolver on X X^T: the same projector L L^T, the same product L R, and
    the eigenvalues equal to the squared singular values."""
    rng = np.random.default_rng(11)
    for P, d, r in [(8, 8, 3), (32, 64, 8), (64, 128, 16), (64, 128, 24)]:
        # well-separated spectrum around the cut, so the kept subspace is unique
        U, _ = np.linalg.qr(rng.standard_normal((P, P)))
        W, _ = np.linalg.qr(rng.standard_normal((d, P)))
        sig = np.sort(rng.uniform(1.0, 2.0, P))[::-1] * np.where(np.arange(P) < r, 10.0, 1.0)
        X = (U * sig) @ W.T
        L, R, S = oracle.factorize(X, r)
        lam, Q = np.linalg.eigh(X @ X.T)  # ascending
        Qr = Q[:, ::-1][:, :r]
        assert np.allclose(L @ L.T, Qr @ Qr.T, atol=1e-10)
        assert np.allclose(L @ R, Qr @ (Qr.T @ X), atol=1e-10 * sig[0])
        assert np.allclose(S[:r] ** 2, lam[::-1][:r], rtol=1e-10)


def test_two_by_two_closed_form():
    """Singular values of a 2 x d page from the closed-form eigenvalues of
    the 2 x 2 Gram X X^T: (tr +- sqrt(tr^2 - 4 det)) / 2."""
    rng = np.random.default_rng(2)
    for d in (2, 3, 8):
        X = rng.standard_normal((2, d))
        G = X @ X.T
        tr, det = G[0, 0] + G[1, 1], G[0, 0] * G[1, 1] - G[0, 1] ** 2
        disc = math.sqrt(max(tr * tr - 4 * det, 0.0))
        lam = np.array([(tr + disc) / 2, (tr - disc) / 2])
        _, S, _, _ = oracle.svd(X)
        assert np.allclose(S ** 2, lam, rtol=1e-12, atol=1e-12 * tr)


def _best_sampled_error(X, r, samples, rng):
    """Smallest ||X - Q Q^T X||^2 over random orthonormal P x r frames Q."""
    P = X.shape[0]
    best = np.inf
    for _ in range(samples):
        Q, _ = np.linalg.qr(rng.standard_normal((P, r)))
        best = min(best, np.sum((X - Q @ (Q.T @ X)) ** 2))
    return best


@pytest.mark.parametrize("r", [1, 2])
def test_brute_force_4x4(r):
    """Eckart-Young on 4 x 4 pages by brute force over frames on the sphere:
    no sampled rank-r projection beats the oracle, and the sampled minimum,
    refined by alternating projection from its frame, reaches it."""
    rng = np.random.default_rng(3 + r)
    for _ in range(4):
        X = rng.standard_normal((4, 4))
        L, R, S = oracle.factorize(X, r)
        opt = np.sum((X - L @ R) ** 2)
        best = _best_sampled_error(X, r, 20000, rng)
        assert best >= opt * (1 - 1e-12)
        assert best <= opt + 0.05 * np.sum(X ** 2)
        # local refinement: orthogonal iteration started from a random frame
        Q, _ = np.linalg.qr(rng.standard_normal((4, r)))
        for _ in range(2000):
            Q, _ = np.linalg.qr(X @ (X.T @ Q))
        refined = np.sum((X - Q @ (Q.T @ X)) ** 2)
        assert abs(refined - opt) <= 1e-9 * np.sum(X ** 2)


def test_degenerate_pages():
    """All-zero page: zero factors, orthonormal L; rank-1 page: exact at r=1."""
    X = np.zeros((8, 16))
    L, R, S = oracle.factorize(X, 3)
    assert np.all(S == 0) and np.all(R == 0)
    assert np.abs(L.T @ L - np.eye(3)).max() == 0
    rng = np.random.default_rng(4)
    u, v = rng.standard_normal(8), rng.standard_normal(16)
    X = np.outer(u, v)
    L, R, S = oracle.factorize(X, 1)
    assert np.abs(X - L @ R).max() < 1e-12 * np.abs(X).max()
    assert abs(S[0] - np.linalg.norm(u) * np.linalg.norm(v)) < 1e-12 * S[0]


def test_planted_factor_mistakes_are_caught():
    X = _page(32, 64, 5)
    r = 8
    L, R, S = oracle.factorize(X, r)
    L_drop = L.copy(); L_drop[:, 3] = 0.0                   # dropped column
    assert eckart_young_defect(X, L_drop, R, S, r) > 1e-6
    R_sign = R.copy(); R_sign[2] *= -1.0                     # wrong sign
    assert eckart_young_defect(X, L, R_sign, S, r) > 1e-6
    L_perm = L[:, ::-1].copy()                               # wrong index order
    assert eckart_young_defect(X, L_perm, R, S, r) > 1e-6
    L_bad = L + 1e-3 * np.random.default_rng(0).standard_normal(L.shape)
    assert orthonormality_defect(L_bad, R, S, r) > 1e-6


# ---------------------------------------------------------- attention pins

def test_attention_special_cases():
    rng = np.random.default_rng(6)
    d = 16
    q = rng.standard_normal((3, d))
    # one key: softmax of a single score is 1
    K1, V1 = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    assert np.allclose(oracle.attention(q, K1, V1), np.repeat(V1, 3, 0), rtol=0, atol=1e-15)
    # identical keys: uniform weights, output is the mean value row
    K = np.repeat(rng.standard_normal((1, d)), 7, 0)
    V = rng.standard_normal((7, d))
    assert np.allclose(oracle.attention(q, K, V), np.repeat(V.mean(0, keepdims=True), 3, 0), atol=1e-14)
    # two keys: logistic weight of the score difference, scores scaled by 1/sqrt(d)
    K2, V2 = rng.standard_normal((2, d)), rng.standard_normal((2, d))
    out = oracle.attention(q, K2, V2)
    for g in range(3):
        s = K2 @ q[g] / math.sqrt(d)
        w = 1.0 / (1.0 + math.exp(s[1] - s[0]))
        assert np.allclose(out[g], w * V2[0] + (1 - w) * V2[1], atol=1e-14)
    # a dominant key takes all the weight
    Kd = np.zeros((5, d)); Kd[2] = q[0] * 1e4
    Vd = rng.standard_normal((5, d))
    assert np.allclose(oracle.attention(q[:1], Kd, Vd)[0], Vd[2], atol=1e-12)
    # permuting tokens leaves the output unchanged
    K5, V5 = rng.standard_normal((9, d)), rng.standard_normal((9, d))
    perm = rng.permutation(9)
    assert np.allclose(oracle.attention(q, K5, V5), oracle.attention(q, K5[perm], V5[perm]), atol=1e-14)


def test_planted_missing_scale_is_caught():
    rng = np.random.default_rng(7)
    d = 64
    q, K, V = rng.standard_normal((2, d)), rng.standard_normal((2, d)), rng.standard_normal((2, d))
    out = oracle.attention(q, K, V)
    unscaled = oracle.attention(q * math.sqrt(d), K, V)  # as if 1/sqrt(d) were dropped
    s = K @ q[0] / math.sqrt(d)
    w = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    ref = w * V[0] + (1 - w) * V[1]
    assert np.allclose(out[0], ref, atol=1e-14)
    assert not np.allclose(unscaled[0], ref, atol=1e-6)


def _cache(T, P, d, G, r, seed, window=64, sink=4):
    spec = synth.KVSpec(layers=1, kv_heads=1, head_dim=d, page_size=P, inner_rank=6,
                        n_outliers=2, dtype=torch.float32)
    K, V = synth.prefill_kv(spec, T, seq=seed)
    K, V = K[0, 0].double().numpy(), V[0, 0].double().numpy()
    q = synth.queries(1, G, d, step=seed, dtype=torch.float32)[0].double().numpy()
    kinds = oracle.page_kinds(T, P, sink, window)
    n = len(kinds)
    LK = np.zeros((n, P, r)); RK = np.zeros((n, r, d))
    LV = np.zeros((n, P, r)); RV = np.zeros((n, r, d))
    for p in range(n):
        if kinds[p] == oracle.FACTORED:
            LK[p], RK[p], _ = oracle.factorize(K[p * P:(p + 1) * P], r)
            LV[p], RV[p], _ = oracle.factorize(V[p * P:(p + 1) * P], r)
    return q, K, V, kinds, LK, RK, LV, RV


def test_full_rank_factorized_attention_equals_dense():
    """r = min(P, d): every factorized page reconstructs exactly, so mixed
    attention equals dense attention (§3.3 ④ with eq. (2) at full rank)."""
    T, P, d, G = 300, 32, 64, 4
    q, K, V, kinds, LK, RK, LV, RV = _cache(T, P, d, G, r=P, seed=11)
    assert (kinds == oracle.FACTORED).sum() >= 4
    mixed = oracle.decode_head(q, kinds, K, V, LK, RK, LV, RV, T, P)
    dense = oracle.attention(q, K, V)
    assert np.abs(mixed - dense).max() <= 1e-6 * np.abs(dense).max()
    assert np.abs(mixed - dense).max() <= 1e-12 * np.abs(dense).max()


def test_low_rank_attention_uses_reconstruction():
    """At r < P the mixed result equals dense attention over the rows L R
    rebuilt by hand (page-by-page products)."""
    T, P, d, G, r = 200, 32, 64, 4, 8
    q, K, V, kinds, LK, RK, LV, RV = _cache(T, P, d, G, r=r, seed=12)
    Kh, Vh = K.copy(), V.copy()
    for p in np.nonzero(kinds == oracle.FACTORED)[0]:
        Kh[p * P:(p + 1) * P] = LK[p] @ RK[p]
        Vh[p * P:(p + 1) * P] = LV[p] @ RV[p]
    mixed = oracle.decode_head(q, kinds, K, V, LK, RK, LV, RV, T, P)
    assert np.abs(mixed - oracle.attention(q, Kh, Vh)).max() <= 1e-12 * np.abs(mixed).max()
    # a transposed factor or a skipped page changes the result
    LKt = LK.copy(); f = int(np.nonzero(kinds == oracle.FACTORED)[0][0])
    LKt[f] = LKt[f][::-1]
    assert np.abs(oracle.decode_head(q, kinds, K, V, LKt, RK, LV, RV, T, P) - mixed).max() > 1e-6


# ------------------------------------------------------ classification pins

def token_level_kinds(T, P, sink, W):
    """Re-derivation by tokens: a token is dense if it is among the first
    `sink` tokens or the last W; a page is dense if it holds a dense token or
    is incomplete (§3.3 ①②③: sink page, local window, page still filling)."""
    dense_tok = [(t < sink) or (t >= T - W) for t in range(T)]
    kinds = []
    for p in range((T + P - 1) // P):
        toks = range(p * P, min((p + 1) * P, T))
        incomplete = len(toks) < P
        kinds.append(oracle.DENSE if incomplete or any(dense_tok[t] for t in toks) else oracle.FACTORED)
    return np.array(kinds, dtype=np.int32)


def test_classification_exhaustive():
    for P, sink, W in itertools.product((4, 32, 64), (0, 4, 64), (0, 64, 128)):
        for T in range(1, 700):
            assert np.array_equal(oracle.page_kinds(T, P, sink, W), token_level_kinds(T, P, sink, W)), (T, P, sink, W)


@pytest.mark.parametrize("T,P,sink,W,dense", [
    (1024, 32, 4, 64, [0, 30, 31]),          # tiny shape
    (32768, 64, 4, 128, [0, 510, 511]),      # 32K context, P = 64
    (131072, 64, 4, 128, [0, 2046, 2047]),   # 128K context, P = 64
    (32769, 64, 4, 128, [0, 510, 511, 512]),
    (32832, 64, 4, 128, [0, 511, 512]),      # page 510 has left the window
])
def test_classification_config_values(T, P, sink, W, dense):
    kinds = oracle.page_kinds(T, P, sink, W)
    assert list(np.nonzero(kinds == oracle.DENSE)[0]) == dense


# ---------------------------------------------------- printed-value pins

def test_printed_storage_ratios():
    g = json.load(open(GOLDEN))
    c = g["storage_ratio_default"]
    ratio = oracle.page_storage_ratio(c["P"], c["d"], c["rk"], c["rv"])
    assert round(ratio, c["printed_digits"]) == c["printed"]
    a = g["storage_ratio_page_size_ablation"]
    for P, rk, rv in a["configs"]:
        # "near 63%" printed to whole percent: within half a percent point
        assert abs(100 * oracle.page_storage_ratio(P, a["d"], rk, rv) - a["printed_percent"]) <= 0.5 + 1e-9


def test_printed_footprint_and_kv_size():
    g = json.load(open(GOLDEN))
    f = g["steady_state_footprint"]
    n_pages = f["T"] // f["P"]
    rho = oracle.page_storage_ratio(f["P"], f["d"], f["rk"], f["rv"])
    footprint = ((n_pages - f["dense_pages"]) * rho + f["dense_pages"]) / n_pages
    assert abs(100 * footprint - f["printed_percent"]) < 0.02
    assert abs(100 * (footprint - rho) - f["printed_gap_pp"]) < 0.02
    s = g["dense_kv_size"]
    nbytes = oracle.dense_kv_elements(s["layers"], s["kv_heads"], s["T"], s["d"]) * s["bytes_per_element"]
    assert nbytes / 2 ** 30 == s["printed_gib"]


def test_exactly_rank_deficient_pages_converge():
    """Repeated rows, a single constant channel, bf16-rounded rank-1 pages:
    exact rank deficiency must not stall the sweeps, and the pins still hold."""
    rng = np.random.default_rng(8)
    pages = []
    X = np.zeros((64, 128)); X[:, 5] = 3.0; pages.append(X)
    X = rng.standard_normal((64, 128)); X[32:] = X[:32]; pages.append(X)
    u, w = rng.standard_normal(64), rng.standard_normal(128)
    pages.append(torch.from_numpy(np.outer(u, w)).to(torch.bfloat16).double().numpy())
    X = pages[-1].copy(); X[10:] = 0; pages.append(X)
    for X in pages:
        for r in (1, 16):
            L, R, S = oracle.factorize(X, r)
            assert eckart_young_defect(X, L, R, S, r) < 1e-12
            assert np.abs(L.T @ L - np.eye(r)).max() < 1e-12
            ref = np.linalg.svd(X, compute_uv=False)
            assert np.abs(S - ref).max() <= 1e-12 * ref[0]


# ---------------------------------------------------- INT4 factors [PuzzleKV §4.3]

def test_int4_quantization_bounds_and_levels():
    """Every element within half a scale of its level; codes in [-7, 7]; the
    largest magnitude of each group lands on +-7 exactly; zero groups stay zero;
    brute force: each code is the nearest of the 15 symmetric levels."""
    rng = np.random.default_rng(11)
    for per_row in (True, False):
        x = rng.standard_normal((9, 13)) * rng.uniform(0.1, 10.0, size=(9, 1))
        x[3] = 0.0 if per_row else x[3]
        if not per_row:
            x[:, 4] = 0.0
        c, s = oracle.quantize_int4(x, per_row)
        xd = oracle.dequantize_int4(c, s, per_row)
        sc = s[:, None] if per_row else s[None, :]
        assert np.all(np.abs(x - xd) <= sc / 2 * (1 + 1e-12) + 1e-300)
        assert c.min() >= -7 and c.max() <= 7
        groups = x if per_row else x.T
        codes = c if per_row else c.T
        for g, cg, sg in zip(groups, codes, s):
            if np.all(g == 0):
                assert sg == 0 and np.all(cg == 0)
                continue
            assert sg == pytest.approx(np.abs(g).max() / 7, rel=1e-15)
            k = np.argmax(np.abs(g))
            assert abs(int(cg[k])) == 7 and np.sign(cg[k]) == np.sign(g[k])
            levels = np.arange(-7, 8) * sg
            nearest = np.abs(g[:, None] - levels[None, :]).argmin(axis=1) - 7
            assert np.array_equal(nearest, cg)


def test_int4_symmetric_and_scale_invariant():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((16, 24))
    for per_row in (True, False):
        c, s = oracle.quantize_int4(x, per_row)
        cn, sn = oracle.quantize_int4(-x, per_row)
        assert np.array_equal(cn, -c) and np.array_equal(sn, s)  # symmetric: no zero point
        c2, s2 = oracle.quantize_int4(4.0 * x, per_row)          # exact power-of-two scaling
        assert np.array_equal(c2, c) and np.allclose(s2, 4.0 * s, rtol=0, atol=0)


def test_int4_absorption_keeps_the_product():
    """Lt Rt = L R; the j-th column of Lt and row of Rt both have norm
    sqrt(sigma_j) (from the fp64 SVD); absorbing sigma instead of sigma^{1/2}
    into L would break the column norms."""
    X = _page(64, 128, seed=13, k=12, n_out=4)
    r = 16
    L, R, S = oracle.factorize(X, r)
    Lt, Rt = oracle.absorb_sigma(L, R)
    assert np.abs(Lt @ Rt - L @ R).max() <= 1e-12 * np.abs(L @ R).max()
    assert np.allclose(np.linalg.norm(Lt, axis=0), np.sqrt(S[:r]), rtol=1e-12)
    assert np.allclose(np.linalg.norm(Rt, axis=1), np.sqrt(S[:r]), rtol=1e-12)
    wrong = L * S[:r]  # planted mistake: the whole of Sigma on L
    assert not np.allclose(np.linalg.norm(wrong, axis=0), np.sqrt(S[:r]), rtol=1e-6)


def test_printed_int4_storage_ratio():
    """0.187 printed for PuzzleKV + INT4 at 16K (Table 3 setting): the whole
    cache, with the two dense pages of the §4.1 region, at fp16 scales."""
    g = json.load(open(GOLDEN))["storage_ratio_int4"]
    n_pages = g["T"] // g["P"]
    rho4 = oracle.int4_page_storage_ratio(g["P"], g["d"], g["rk"], g["rv"])
    whole = ((n_pages - g["dense_pages"]) * rho4 + g["dense_pages"]) / n_pages
    assert round(whole, g["printed_digits"]) == g["printed"]
    # fp32 scales would not reproduce the printed value
    rho32 = oracle.int4_page_storage_ratio(g["P"], g["d"], g["rk"], g["rv"], scale_bytes=4)
    assert round(((n_pages - g["dense_pages"]) * rho32 + g["dense_pages"]) / n_pages, 3) != g["printed"]


# --- RoPE at cache access for keys factorized before it [PuzzleKV §4.1, Appendix D.3] ---

def _rope_complex(X, pos, theta):
    """Rotate-half RoPE as complex multiplication: z_i = x_i + i x_{i+d/2} turns by pos theta^(-2i/d)."""
    d = X.shape[1]
    h = d // 2
    z = (X[:, :h] + 1j * X[:, h:]) * np.exp(1j * np.outer(pos, theta ** (-2.0 * np.arange(h) / d)))
    return np.concatenate([z.real, z.imag], axis=1)


def test_rope_is_complex_multiplication():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((7, 16))
    pos = np.array([0, 1, 5, 17, 1000, 32767, 131071])
    for theta in (1e4, 5e5):
        got = oracle.rope(X, pos, theta)
        assert np.allclose(got, _rope_complex(X, pos, theta), rtol=0, atol=1e-9)
    assert np.array_equal(oracle.rope(X[:1], [0], 1e4), X[:1])  # position 0 is the identity


def test_rope_relative_position_and_norm():
    """<R(m) q, R(n) k> = <q, R(n - m) k>, and every rotation keeps norms."""
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((1, 128)), rng.standard_normal((1, 128))
    for m, n in ((0, 9), (300, 1000), (40000, 40063)):
        lhs = (oracle.rope(q, [m], 5e5) @ oracle.rope(k, [n], 5e5).T).item()
        rhs = (q @ oracle.rope(k, [n - m], 5e5).T).item()
        assert abs(lhs - rhs) <= 1e-9 * max(1.0, abs(rhs))
        assert np.isclose(np.linalg.norm(oracle.rope(k, [n], 5e5)), np.linalg.norm(k), rtol=1e-13)


def test_prerope_decode_full_rank_is_dense_rope_attention():
    """With keys kept exactly (rank = P), the pre-RoPE hybrid decode is softmax
    attention over the RoPE-rotated keys, stated here independently (complex
    rotation, numpy softmax); at a lower rank it is not."""
    rng = np.random.default_rng(5)
    T, P, d, G, theta = 230, 32, 64, 3, 1e4
    K, V = rng.standard_normal((T, d)), rng.standard_normal((T, d))
    q = rng.standard_normal((G, d)) / np.sqrt(d)
    kinds = oracle.page_kinds(T, P, 4, 64)
    n = len(kinds)

    def factors(X, r):
        L, R = np.zeros((n, P, r)), np.zeros((n, r, d))
        for p in np.nonzero(kinds == oracle.FACTORED)[0]:
            L[p], R[p], _ = oracle.factorize(X[p * P:(p + 1) * P], r)
        return L, R

    Kr = _rope_complex(K, np.arange(T), theta)
    s = q @ Kr.T / np.sqrt(d)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    want = (w / w.sum(axis=1, keepdims=True)) @ V
    LK, RK = factors(K, P)
    LV, RV = factors(V, P)
    got = oracle.decode_head_rope(q, kinds, K, V, LK, RK, LV, RV, T, P, theta)
    assert np.max(np.abs(got - want)) <= 1e-10
    LK, RK = factors(K, 8)
    low = oracle.decode_head_rope(q, kinds, K, V, LK, RK, LV, RV, T, P, theta)
    assert np.max(np.abs(low - want)) > 1e-3
    # keys rotated after their reconstruction, not before the factorization
    # (a reading error this path must not make)
    post = oracle.decode_head(q, kinds, Kr, V, *factors(Kr, 8), LV, RV, T, P)
    assert np.max(np.abs(post - low)) > 1e-4


def test_batched_wrapper_equals_per_page():
    """The batched oracle wrapper (independent pages on several host threads,
    [PuzzleKV §3.3 ③]) gives, page for page, exactly the pinned single-page
    factorization: a stride or offset mistake in the wrapper would move some
    page's factors onto another page's slot."""
    P, d, r = 32, 64, 8
    X = np.stack([_page(P, d, seed=s) for s in range(21)])
    X[5] = 0.0                              # all-zero page (C12)
    X[9] = np.outer(X[9][:, 0], X[9][0])    # exactly rank one
    ref = [oracle.factorize(X[i], r) for i in range(X.shape[0])]
    for nthreads in (1, 4):
        L, R, S = oracle.factorize_pages(X, r, nthreads)
        for i, (Li, Ri, Si) in enumerate(ref):
            assert np.array_equal(L[i], Li) and np.array_equal(R[i], Ri) and np.array_equal(S[i], Si), (nthreads, i)
    # a wrapper that paired pages with the wrong slots would fail the comparison
    L, R, S = oracle.factorize_pages(X[::-1].copy(), r, 4)
    assert not np.array_equal(L[0] @ R[0], ref[0][0] @ ref[0][1])
