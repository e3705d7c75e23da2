"""Seeded synthetic inputs shaped like the KV caches the PuzzleKV page describes.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It draws random numbers and arranges them; it holds none of the
compression method's arithmetic (no factorization, no attention).

Generator recipe (stated once here, used everywhere):

* A cache of ``T`` tokens is cut into ``ceil(T / P)`` pages of ``P`` tokens.
  Each page of each (layer, KV head, K/V) is ``0.5 * A @ B + 0.05 * N`` with
  ``A`` (P x k), ``B`` (k x d) and ``N`` (P x d) i.i.d. N(0, 1), drawn fresh per
  page (``k`` = inner rank: 6 for the tiny case, 12 otherwise).
* ``n_out`` outlier channels per (layer, KV head, K/V) are drawn once with a
  seeded permutation; those whole columns (signal and noise) are scaled by 8
  in every page.
* Optional RoPE on keys (half-split "rotate-half" pairing ``(i, i + d/2)``,
  ``theta_i = base ** (-2 i / d)``) at absolute positions, applied before the
  keys reach the cache (post-RoPE keys, as in PuzzleKV §4.2).
* Queries are N(0, 1) / sqrt(d).
* Seeds: K of layer ``l`` in sequence ``b`` uses ``42 + 2 l + 10007 b``, V uses
  that plus one; decode-phase pages use their own per-page seed so that
  tokens appended during decoding come from the same low-rank-plus-noise
  model; queries use ``10**6 + 1000 * step + layer``; ragged batch lengths
  use seed 7.  42 is the seed the PuzzleKV page states for its evaluations
  (Appendix A.1).
"""
from .generators import (  # noqa: F401
    KVSpec,
    kv_seed,
    outlier_channels,
    prefill_kv,
    decode_page,
    decode_tokens,
    decode_rows,
    queries,
    batch_lengths,
    apply_rope,
)
