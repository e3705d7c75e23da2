"""PuzzleKV oracle: plain, slow, fp64 CPU reference of the hot path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product
library (``page_wise_rank_gb300``) never does, and the oracle never imports
the product.  The arithmetic lives in ``puzzlekv_oracle.c``; this module only
marshals numpy arrays (fp64) through ctypes and states the closed-form byte
formulas of the page.

Citations name sections/equations of "PuzzleKV: Page-Wise Low-Rank
Decomposition for KV Cache Compression" ([PuzzleKV]).

Pins (see tests/test_oracle_pins.py): Eckart-Young energy identity,
orthonormal factors, singular values against LAPACK, the Gram route
(top-r eigenvectors of X X^T from LAPACK's symmetric eigensolver give the
same L L^T and L R), 2x2 closed form,
brute force over the unit sphere on 4x4 pages, full-rank factorized
attention equal to dense attention, closed-form attention special cases,
token-level reclassification, the page's printed storage ratios, and RoPE
against complex multiplication and its relative-position property.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

FACTORED = 0
DENSE = 1

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        L.oracle_page_kinds.argtypes = [ctypes.c_int] * 4 + [ip, ctypes.c_int]
        L.oracle_page_kinds.restype = ctypes.c_int
        L.oracle_svd.argtypes = [dp, ctypes.c_int, ctypes.c_int, dp, dp, dp]
        L.oracle_svd.restype = ctypes.c_int
        L.oracle_factorize_page.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp]
        L.oracle_factorize_page.restype = ctypes.c_int
        L.oracle_factorize_pages.argtypes = [dp, ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             dp, dp, dp, ctypes.c_int]
        L.oracle_factorize_pages.restype = ctypes.c_int
        L.oracle_attention.argtypes = [dp, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp]
        L.oracle_attention.restype = None
        L.oracle_decode_head.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ip,
                                         dp, dp, dp, dp, ctypes.c_int, dp, dp, ctypes.c_int, dp]
        L.oracle_decode_head.restype = None
        cp = ctypes.POINTER(ctypes.c_byte)
        L.oracle_absorb_sigma.argtypes = [dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp]
        L.oracle_absorb_sigma.restype = None
        L.oracle_quantize_int4.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, cp, dp]
        L.oracle_quantize_int4.restype = None
        L.oracle_dequantize_int4.argtypes = [cp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp]
        L.oracle_rope.argtypes = [dp, ctypes.POINTER(ctypes.c_long), ctypes.c_long, ctypes.c_int, ctypes.c_double, dp]
        L.oracle_rope.restype = None
        L.oracle_dequantize_int4.restype = None
        _lib = L
    return _lib


def _f64(a) -> np.ndarray:
    """Exact upcast of the stored values (bf16/fp32 torch tensors or arrays) to fp64."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def page_kinds(T: int, P: int, sink_tokens: int, window_tokens: int) -> np.ndarray:
    """Kind (FACTORED=0 / DENSE=1) of each of the ceil(T/P) pages [PuzzleKV §3.3 ①②③, ⑤]."""
    n = (T + P - 1) // P
    out = np.zeros(max(n, 1), dtype=np.int32)
    got = lib().oracle_page_kinds(T, P, sink_tokens, window_tokens,
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), out.size)
    assert got == n
    return out[:n]


def svd(X):
    """X (n x d, n <= d) = U diag(S) W^T by one-sided Jacobi; returns (U, S, Y, sweeps)
    with Y = diag(S) W^T [PuzzleKV §3.2 Truncated SVD]."""
    X = _f64(X)
    n, d = X.shape
    U = np.zeros((n, n))
    S = np.zeros(n)
    Y = np.zeros((n, d))
    sweeps = lib().oracle_svd(_p(X), n, d, _p(U), _p(S), _p(Y))
    return U, S, Y, sweeps


def factorize(X, r: int):
    """Rank-r factors of one page: L = U_r (P x r), R = Sigma_r W_r^T (r x d),
    plus all singular values [PuzzleKV §3.3 eq. (2)]."""
    X = _f64(X)
    P, d = X.shape
    L = np.zeros((P, r))
    R = np.zeros((r, d))
    S = np.zeros(P)
    st = lib().oracle_factorize_page(_p(X), P, d, r, _p(L), _p(R), _p(S))
    if st < 0:
        raise RuntimeError("oracle SVD did not converge")
    return L, R, S


def factorize_pages(X, r: int, nthreads: int = 1):
    """Batched rank-r factors of X[n, P, d] -> L[n, P, r], R[n, r, d], S[n, P]."""
    X = _f64(X)
    n, P, d = X.shape
    L = np.zeros((n, P, r))
    R = np.zeros((n, r, d))
    S = np.zeros((n, P))
    bad = lib().oracle_factorize_pages(_p(X), n, P, d, r, _p(L), _p(R), _p(S), nthreads)
    if bad:
        raise RuntimeError(f"oracle SVD did not converge on {bad} pages")
    return L, R, S


def attention(q, K, V) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V for q [G, d], K, V [T, d] [PuzzleKV §3.2 eq. (1)]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    G, d = q.shape
    T = K.shape[0]
    out = np.zeros((G, d))
    lib().oracle_attention(_p(q), _p(K), _p(V), G, T, d, _p(out))
    return out


def decode_head(q, kinds, Kd, Vd, LK, RK, LV, RV, T: int, P: int) -> np.ndarray:
    """Attention of G query rows over one KV head's hybrid cache: factorized
    pages reconstructed as L R, dense pages as stored [PuzzleKV §3.3 ④].

    kinds [n_pages]; Kd, Vd [>= T, d]; LK [n_pages, P, rk]; RK [n_pages, rk, d];
    LV [n_pages, P, rv]; RV [n_pages, rv, d].
    """
    q = _f64(q)
    G, d = q.shape
    kinds = np.ascontiguousarray(np.asarray(kinds, dtype=np.int32))
    Kd, Vd, LK, RK, LV, RV = (_f64(a) for a in (Kd, Vd, LK, RK, LV, RV))
    n_pages = (T + P - 1) // P
    assert kinds.shape[0] >= n_pages and Kd.shape[0] >= T and Vd.shape[0] >= T
    rk, rv = LK.shape[-1], LV.shape[-1]
    assert LK.shape[0] >= n_pages and RK.shape[0] >= n_pages
    out = np.zeros((G, d))
    lib().oracle_decode_head(_p(q), G, d, T, P, kinds.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                             _p(Kd), _p(Vd), _p(LK), _p(RK), rk, _p(LV), _p(RV), rv, _p(out))
    return out


def rope(X, positions, theta: float) -> np.ndarray:
    """Rotary position embedding of the rows of X [n, d] at `positions` (rotate-half
    pairing (i, i + d/2), angle position * theta^(-2i/d)) [PuzzleKV §4.1, Appendix D.3]."""
    X = np.ascontiguousarray(_f64(X))
    n, d = X.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    assert pos.shape == (n,) and d % 2 == 0
    out = np.zeros_like(X)
    lib().oracle_rope(_p(X), pos.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), n, d, float(theta), _p(out))
    return out


def decode_head_rope(q, kinds, Kd, Vd, LK, RK, LV, RV, T: int, P: int, theta: float) -> np.ndarray:
    """decode_head for keys stored before RoPE: every key is reconstructed as
    stored (dense rows, or L_K R_K of its page), turned by RoPE at its absolute
    position, and the query rows (already rotated at their own position)
    attend with plain softmax [PuzzleKV §3.3 ④, §4.1, Appendix D.3]."""
    kinds = np.asarray(kinds)
    Kd, Vd, LK, RK, LV, RV = (_f64(a) for a in (Kd, Vd, LK, RK, LV, RV))
    K = Kd[:T].copy()
    V = Vd[:T].copy()
    for p in range((T + P - 1) // P):
        if kinds[p] == FACTORED:
            K[p * P:(p + 1) * P] = LK[p] @ RK[p]
            V[p * P:(p + 1) * P] = LV[p] @ RV[p]
    return attention(q, rope(K, np.arange(T), theta), V)


def absorb_sigma(L, R):
    """(Lt, Rt) = (U_r Sigma^{1/2}, Sigma^{1/2} W_r^T) from the eq. (2) factors
    L = U_r, R = Sigma_r W_r^T [PuzzleKV §4.3]."""
    L, R = _f64(L), _f64(R)
    P, r = L.shape
    d = R.shape[1]
    Lt, Rt = np.empty_like(L), np.empty_like(R)
    lib().oracle_absorb_sigma(_p(L), _p(R), P, d, r, _p(Lt), _p(Rt))
    return Lt, Rt


def quantize_int4(x, per_row: bool):
    """Symmetric INT4 codes (int8 array, values in [-7, 7]) and fp64 scales,
    one per row (per_row) or per column [PuzzleKV §4.3]."""
    x = _f64(x)
    rows, cols = x.shape
    codes = np.empty((rows, cols), dtype=np.int8)
    scales = np.empty(rows if per_row else cols, dtype=np.float64)
    lib().oracle_quantize_int4(_p(x), rows, cols, int(per_row), codes.ctypes.data_as(ctypes.POINTER(ctypes.c_byte)),
                               _p(scales))
    return codes, scales


def dequantize_int4(codes, scales, per_row: bool) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    scales = _f64(scales)
    rows, cols = codes.shape
    x = np.empty((rows, cols), dtype=np.float64)
    lib().oracle_dequantize_int4(codes.ctypes.data_as(ctypes.POINTER(ctypes.c_byte)), _p(scales), rows, cols,
                                 int(per_row), _p(x))
    return x


# which factor is quantized per row [PuzzleKV §4.3]: column-wise for L_K, R_K
# and R_V, row-wise for L_V (factors in the eq. (2) orientation: L is P x r,
# R is r x d)
INT4_PER_ROW = {"LK": False, "RK": False, "LV": True, "RV": False}


def int4_page_storage_ratio(P: int, d: int, rk: int, rv: int, scale_bytes: int = 2) -> float:
    """Bytes of one page's INT4 key and value factors (4-bit codes plus one
    scale per quantization group: r_K + d for the key, P + d for the value)
    over the dense page pair's bf16 bytes [PuzzleKV §4.3]."""
    codes = ((P + d) * rk + (P + d) * rv) / 2.0
    scales = scale_bytes * ((rk + d) + (P + d))
    return (codes + scales) / (2.0 * P * d * 2)


def page_storage_ratio(P: int, d: int, rk: int, rv: int) -> float:
    """Storage of a factorized key-value page pair relative to dense, eq. (3) / (6):
    (rK + rV)(P + d) / (2 P d) [PuzzleKV §3.3 eq. (3); Appendix D.1 eq. (6)]."""
    return (rk + rv) * (P + d) / (2.0 * P * d)


def dense_kv_elements(layers: int, kv_heads: int, T: int, d: int) -> int:
    """Elements a single request's dense KV cache holds: 2 L H_kv T d [PuzzleKV §1]."""
    return 2 * layers * kv_heads * T * d
