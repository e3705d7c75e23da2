"""Seeded generators for synthetic KV caches, decode-phase tokens and queries.

Everything here is random-number drawing and arrangement; see the package
docstring for the recipe.  Works on any torch device: CPU for tests that feed
the CPU oracle, CUDA for full-size workloads (where the oracle then reads
sampled pages copied back to the host).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Optional, Sequence, Tuple

import torch


@dataclass(frozen=True)
class KVSpec:
    """Shape of one synthetic cache (per sequence)."""

    layers: int
    kv_heads: int
    head_dim: int
    page_size: int
    inner_rank: int = 12
    n_outliers: int = 4
    rope_base: Optional[float] = None
    dtype: torch.dtype = torch.bfloat16


def kv_seed(layer: int, kind: int, seq: int = 0) -> int:
    """Seed of the prefill pages of (layer, K=0 / V=1, sequence)."""
    return 42 + 2 * layer + kind + 10007 * seq


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def outlier_channels(spec: KVSpec, layer: int, kind: int, seq: int = 0) -> torch.Tensor:
    """[H, n_outliers] distinct channel indices per KV head (drawn on the CPU,
    so CPU and CUDA runs see the same channels)."""
    g = _generator(kv_seed(layer, kind, seq) + 900_000_000, "cpu")
    rows = [torch.randperm(spec.head_dim, generator=g)[: spec.n_outliers]
            for _ in range(spec.kv_heads)]
    return torch.stack(rows) if rows else torch.zeros(0, spec.n_outliers, dtype=torch.long)


def apply_rope(x: torch.Tensor, positions: torch.Tensor, base: float) -> torch.Tensor:
    """Half-split rotary embedding on the last dim of ``x`` ([..., T, d]) at
    absolute ``positions`` ([T]); pairs channel i with i + d/2."""
    d = x.shape[-1]
    half = d // 2
    inv = base ** (-torch.arange(half, dtype=torch.float64, device=x.device) * 2.0 / d)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]
    cos = torch.cos(ang).to(torch.float32)
    sin = torch.sin(ang).to(torch.float32)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def _scale_outliers(x: torch.Tensor, chans: torch.Tensor) -> torch.Tensor:
    # x: [H, T, d]; chans: [H, n_out]
    if chans.numel() == 0:
        return x
    scale = torch.ones(x.shape[0], x.shape[-1], dtype=x.dtype, device=x.device)
    scale.scatter_(1, chans.to(x.device), 8.0)
    return x * scale[:, None, :]


def _pages(g: torch.Generator, spec: KVSpec, heads: int, n_pages: int, device) -> torch.Tensor:
    """[heads, n_pages * P, d] fp32 low-rank-plus-noise rows."""
    P, d, k = spec.page_size, spec.head_dim, spec.inner_rank
    a = torch.randn(heads, n_pages, P, k, generator=g, device=device)
    b = torch.randn(heads, n_pages, k, d, generator=g, device=device)
    n = torch.randn(heads, n_pages, P, d, generator=g, device=device)
    x = 0.5 * torch.matmul(a, b) + 0.05 * n
    return x.reshape(heads, n_pages * P, d)


def prefill_kv(spec: KVSpec, T: int, seq: int = 0, device="cpu",
               out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None
               ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Dense prompt cache of one sequence: K, V as [L, H, T, d] in ``spec.dtype``.

    Keys carry RoPE at positions 0..T-1 when ``spec.rope_base`` is set.
    ``out`` may supply preallocated destination tensors.
    """
    L, H, d, P = spec.layers, spec.kv_heads, spec.head_dim, spec.page_size
    n_pg = (T + P - 1) // P
    if out is None:
        K = torch.empty(L, H, T, d, dtype=spec.dtype, device=device)
        V = torch.empty(L, H, T, d, dtype=spec.dtype, device=device)
    else:
        K, V = out
    pos = torch.arange(T, device=device)
    for layer in range(L):
        for kind, dst in ((0, K), (1, V)):
            g = _generator(kv_seed(layer, kind, seq), device)
            x = _pages(g, spec, H, n_pg, device)[:, :T]
            x = _scale_outliers(x, outlier_channels(spec, layer, kind, seq))
            if kind == 0 and spec.rope_base is not None:
                x = apply_rope(x, pos, spec.rope_base)
            dst[layer].copy_(x.to(spec.dtype))
            del x
    return K, V


def decode_page(spec: KVSpec, layer: int, kind: int, seq: int, page: int, device="cpu") -> torch.Tensor:
    """[H, P, d] fp32 page (pre-RoPE) from which decode-phase tokens of
    ``page`` are taken, one row per generated token."""
    g = _generator(kv_seed(layer, kind, seq) * 1_000_003 + 7919 * page + 13, device)
    x = _pages(g, spec, spec.kv_heads, 1, device)
    return _scale_outliers(x, outlier_channels(spec, layer, kind, seq))


def decode_tokens(spec: KVSpec, layer: int, seqs: Sequence[int], positions: Sequence[int],
                  device="cpu", cache: Optional[Dict] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """New (k, v) rows for one decode step: each [B, H, d] in ``spec.dtype``.

    Row ``pos % P`` of the decode page of ``pos // P``; keys get RoPE at
    ``pos``.  ``cache`` (a dict) memoises generated pages across steps.
    """
    P = spec.page_size
    ks, vs = [], []
    for seq, pos in zip(seqs, positions):
        page, row = divmod(int(pos), P)
        rows = []
        for kind in (0, 1):
            key = (layer, kind, seq, page)
            if cache is not None and key in cache:
                pg = cache[key]
            else:
                pg = decode_page(spec, layer, kind, seq, page, device)
                if cache is not None:
                    cache[key] = pg
            x = pg[:, row:row + 1, :]
            if kind == 0 and spec.rope_base is not None:
                x = apply_rope(x, torch.tensor([int(pos)], device=device), spec.rope_base)
            rows.append(x[:, 0, :])
        ks.append(rows[0])
        vs.append(rows[1])
    return (torch.stack(ks).to(spec.dtype), torch.stack(vs).to(spec.dtype))


def decode_rows(spec: KVSpec, layer: int, seq: int, first: int, n: int, device="cpu"
                ) -> Tuple[torch.Tensor, torch.Tensor]:
    """The rows ``decode_tokens`` gives sequence ``seq`` at positions
    first .. first + n - 1, all at once: (K, V), each [H, n, d] in ``spec.dtype``."""
    P = spec.page_size
    p0, p1 = first // P, (first + n - 1) // P
    out = []
    for kind in (0, 1):
        x = torch.cat([decode_page(spec, layer, kind, seq, p, device) for p in range(p0, p1 + 1)], dim=1)
        x = x[:, first - p0 * P: first - p0 * P + n]
        if kind == 0 and spec.rope_base is not None:
            x = apply_rope(x, torch.arange(first, first + n, device=device), spec.rope_base)
        out.append(x.to(spec.dtype))
    return out[0], out[1]


def queries(B: int, Hq: int, d: int, step: int, layer: int = 0, device="cpu",
            dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """[B, Hq, d] queries, N(0, 1) / sqrt(d)."""
    g = _generator(10 ** 6 + 1000 * step + layer, device)
    q = torch.randn(B, Hq, d, generator=g, device=device) / math.sqrt(d)
    return q.to(dtype)


def batch_lengths(B: int, lo: int, hi: int, seed: int = 7) -> list:
    """B context lengths drawn uniformly from [lo, hi] inclusive."""
    g = _generator(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]
