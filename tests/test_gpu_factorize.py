"""GPU parity of batched page factorization against the fp64 oracle.

Tolerance (spec reading C5): per page, the reconstruction error of the
kernel's fp32 factors exceeds the oracle's optimum e* = sqrt(sum_{i>r} s_i^2)
by at most 1e-3 relative.  Factors themselves are never compared
elementwise (singular vectors are unique only up to sign / rotation).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from page_wise_rank_gb300 import build
    build.build()
    import page_wise_rank_gb300 as m
    return m


def pages(n, P, d, dtype, seed=0, k=12, n_out=4, rope=None):
    spec = synth.KVSpec(layers=1, kv_heads=1, head_dim=d, page_size=P, inner_rank=min(k, P), n_outliers=n_out,
                        rope_base=rope, dtype=dtype)
    K, V = synth.prefill_kv(spec, n * P, seq=seed)
    X = torch.cat([K[0, 0], V[0, 0]]).reshape(2 * n, P, d)
    return X


def check_c5(X, L, R, S, r, tol=1e-3):
    worst = 0.0
    Xd = X.double().numpy()
    Ld, Rd = L.double().cpu().numpy(), R.double().cpu().numpy()
    Sg = S.double().cpu().numpy() if S is not None else None
    for i in range(X.shape[0]):
        _, _, So = oracle.factorize(Xd[i], r)
        e_star = math.sqrt(np.sum(So[r:] ** 2))
        e = np.linalg.norm(Xd[i] - Ld[i] @ Rd[i])
        nx = np.linalg.norm(Xd[i])
        if e_star > 1e-6 * nx:
            worst = max(worst, (e - e_star) / e_star)
        else:  # (near) exact rank <= r: measure against the page norm
            worst = max(worst, e / nx)
        # singular values from the fp32 Gram eigenvalues (when requested)
        if Sg is not None:
            assert np.abs(Sg[i] - So).max() <= 2e-4 * So[0] + 1e-6
        # orthonormal left factor
        assert np.abs(Ld[i].T @ Ld[i] - np.eye(r)).max() < 2e-5
    assert worst <= tol, worst
    return worst


@pytest.mark.parametrize("P,d,r", [(64, 128, 16), (64, 128, 24), (64, 128, 1), (64, 128, 32), (64, 128, 40), (32, 128, 16),
                                   (32, 64, 8), (16, 64, 8), (16, 128, 9)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_factorize_batch_c5(pkv, P, d, r, dtype):
    """With and without singular values (with them every eigenvalue is
    computed, without them only the kept ones when r <= P / 2, the store's
    case), on both eigensolver paths (r <= P / 2: bisection and inverse
    iteration; above: QL).  Either way the reconstruction is within C5."""
    X = pages(150, P, d, dtype, seed=P + d + r)
    L, R, S, status = pkv.factorize_batch(X.cuda(), r, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_c5(X, L, R, S, r)
    L2, R2, _, status = pkv.factorize_batch(X.cuda(), r, out_dtype=torch.float32, sigma=False)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_c5(X, L2, R2, None, r)


def test_full_rank_reconstructs(pkv):
    for dtype in (torch.float32, torch.bfloat16):
        X = pages(40, 32, 64, dtype, seed=3, k=6, n_out=2)
        L, R, S, status = pkv.factorize_batch(X.cuda(), 32, out_dtype=torch.float32)
        Xd, rec = X.double(), torch.bmm(L.double(), R.double()).cpu()
        rel = (torch.linalg.norm(Xd - rec, dim=(1, 2)) / torch.linalg.norm(Xd, dim=(1, 2))).max().item()
        assert rel < 1e-5 and int(status.item()) == 0


def test_degenerate_pages(pkv):
    P, d, r = 64, 128, 16
    X = torch.zeros(6, P, d, dtype=torch.bfloat16)
    u = torch.randn(P, generator=torch.Generator().manual_seed(0))
    w = torch.randn(d, generator=torch.Generator().manual_seed(1))
    X[1] = torch.outer(u, w).bfloat16()            # rank 1
    X[2] = X[1]
    X[2, 10:] = 0                                  # rank 1, mostly zero rows
    X[3, :, 5] = 3.0                               # one constant channel
    X[4] = torch.randn(P, d, generator=torch.Generator().manual_seed(2)).bfloat16()
    X[4, 32:] = X[4, :32]                          # repeated rows
    X[5] = pages(1, P, d, torch.bfloat16, seed=9)[0]
    L, R, S, status = pkv.factorize_batch(X.cuda(), r, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.all(R[0] == 0) and torch.isfinite(L).all() and torch.isfinite(R).all()
    Ld = L[0].double().cpu()
    assert (Ld.T @ Ld - torch.eye(r, dtype=torch.float64)).abs().max() < 1e-6
    for i in range(1, 6):
        Xd = X[i].double().numpy()
        _, _, So = oracle.factorize(Xd, r)
        e_star = math.sqrt(np.sum(So[r:] ** 2))
        e = np.linalg.norm(Xd - L[i].double().cpu().numpy() @ R[i].double().cpu().numpy())
        # fp32 floor: the Gram matrix and a backward-stable eigensolve of it
        # carry a few units of fp32 roundoff (u = 2^-23) of ||X||^2 in every
        # eigenvalue, so a page whose discarded energy sits below that can
        # only be matched to it (the rank-1 page: excess 1.9 u ||X||^2)
        assert e ** 2 <= e_star ** 2 * (1 + 2e-3) + 4 * 2.0 ** -23 * np.sum(Xd ** 2), (i, e, e_star)


def test_bf16_output_is_rounded_fp32_output(pkv):
    X = pages(32, 64, 128, torch.bfloat16, seed=5)
    L32, R32, _, _ = pkv.factorize_batch(X.cuda(), 16, out_dtype=torch.float32)
    L16, R16, _, _ = pkv.factorize_batch(X.cuda(), 16, out_dtype=torch.bfloat16)
    assert torch.equal(L32.bfloat16(), L16) and torch.equal(R32.bfloat16(), R16)


def test_rope_keys_llama_shape(pkv):
    """Post-RoPE keys at 32K positions (base 5e5), the 32K-context key pages."""
    spec = synth.KVSpec(layers=1, kv_heads=1, head_dim=128, page_size=64, inner_rank=12, n_outliers=4,
                        rope_base=5e5, dtype=torch.bfloat16)
    K, _ = synth.prefill_kv(spec, 64 * 512)
    X = K[0, 0].reshape(512, 64, 128)[::7].contiguous()
    L, R, S, status = pkv.factorize_batch(X.cuda(), 16, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_c5(X, L, R, S, 16)


def structured_pages(P=64, d=128, seed=3):
    """Valid pages whose Gram matrix drives the eigensolve to its edge cases:
    the trailing columns of the Householder reduction fall to (or towards)
    the subnormal range, or split the tridiagonal exactly."""
    X = pages(2, P, d, torch.float32, seed=seed)[:4].clone()
    X[0, 45:] = X[0, 44]                   # the last 19 rows repeat one row (a decode loop fed one token)
    X[1, 32:] = X[1, 31]                   # half the page one repeated row
    X[2, :P // 2, d // 2:] = 0             # two row blocks on disjoint channels: G is block-diagonal
    X[2, P // 2:, :d // 2] = 0
    X[3, 1:] = X[3, 0]                     # every row the same: rank 1 exactly
    return X.bfloat16()


@pytest.mark.parametrize("r", [16, 24])
def test_structured_pages(pkv, r):
    """Repeated rows, a block-diagonal Gram matrix and an exactly rank-1 page:
    finite, orthonormal factors within the C5 bound (with the fp32 floor of
    test_degenerate_pages), from a launch of a few pages (1024 threads per
    page) and bitwise the same from a launch of 2,800 (256 threads, several
    pages per CTA)."""
    X = structured_pages()
    L, R, S, status = pkv.factorize_batch(X.cuda(), r, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(L).all() and torch.isfinite(R).all() and torch.isfinite(S).all()
    for i in range(X.shape[0]):
        Xd = X[i].double().numpy()
        Ld, Rd = L[i].double().cpu().numpy(), R[i].double().cpu().numpy()
        assert np.abs(Ld.T @ Ld - np.eye(r)).max() < 2e-5, i
        _, _, So = oracle.factorize(Xd, r)
        e_star2 = float(np.sum(So[r:] ** 2))
        e2 = float(np.linalg.norm(Xd - Ld @ Rd) ** 2)
        assert e2 <= e_star2 * (1 + 2e-3) + 4 * 2.0 ** -23 * np.sum(Xd ** 2), (i, e2, e_star2)
    big = X.repeat(700, 1, 1)
    Lb, Rb, _, status = pkv.factorize_batch(big.cuda(), r, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for j in (0, 1, 2, 3, 1401, 2798, 2799):
        assert torch.equal(Lb[j], L[j % 4]) and torch.equal(Rb[j], R[j % 4]), j


def test_large_batch_matches_small_batch(pkv):
    """Many CTAs (a grid-stride over pages) give the same factors as one-page launches."""
    X = pages(400, 64, 128, torch.bfloat16, seed=11)
    L, R, _, _ = pkv.factorize_batch(X.cuda(), 24, out_dtype=torch.float32)
    for i in (0, 1, 399, 799):
        L1, R1, _, _ = pkv.factorize_batch(X[i:i + 1].cuda(), 24, out_dtype=torch.float32)
        assert torch.equal(L1[0], L[i]) and torch.equal(R1[0], R[i])
