"""Helpers shared by the GPU parity tests: build a store from a synthetic
cache, replay decode steps, and compute the oracle's answer on the factors
the GPU stored (decode parity on identical factors)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from store_layout import Layout, descriptors, factor_pool_slice, lengths, read_factors


def rel_err_rows(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max_i |o_i - ref_i| / max_i |ref_i|."""
    got = np.atleast_2d(got)
    ref = np.atleast_2d(ref)
    return float((np.abs(got - ref).max(axis=1) / np.abs(ref).max(axis=1)).max())


class HostCache:
    """Host copy of every key/value row fed to the store, per (seq, layer, head)."""

    def __init__(self):
        self.k = {}
        self.v = {}

    def set_prefill(self, seq, K, V):
        # K, V: [L, H, T, d] (any device)
        K, V = K.detach().cpu(), V.detach().cpu()
        for l in range(K.shape[0]):
            for h in range(K.shape[1]):
                self.k[(seq, l, h)] = [K[l, h]]
                self.v[(seq, l, h)] = [V[l, h]]

    def append(self, seq, layer, k, v):
        # k, v: [H, d]
        k, v = k.detach().cpu(), v.detach().cpu()
        for h in range(k.shape[0]):
            self.k[(seq, layer, h)].append(k[h:h + 1])
            self.v[(seq, layer, h)].append(v[h:h + 1])

    def rows(self, seq, layer, h):
        K = torch.cat(self.k[(seq, layer, h)]).double().numpy()
        V = torch.cat(self.v[(seq, layer, h)]).double().numpy()
        return K, V


def oracle_decode_on_store(store, cfg, host: HostCache, seq: int, layer: int, h: int, q_rows: np.ndarray,
                           fpool=None) -> np.ndarray:
    """Oracle attention of the G query rows of KV head h, run on the factors
    the store holds (copied back and upcast) and the dense rows it was fed."""
    lay = Layout(cfg)
    K, V = host.rows(seq, layer, h)
    T = K.shape[0]
    P = cfg.page_size
    kinds = oracle.page_kinds(T, P, cfg.sink_tokens, cfg.recent_tokens)
    n = len(kinds)
    if fpool is None:
        fpool = factor_pool_slice(store, lay, layer, seq, h)
    LK, RK = np.zeros((n, P, cfg.rank_k)), np.zeros((n, cfg.rank_k, cfg.head_dim))
    LV, RV = np.zeros((n, P, cfg.rank_v)), np.zeros((n, cfg.rank_v, cfg.head_dim))
    for p in np.nonzero(kinds == oracle.FACTORED)[0]:
        LK[p], RK[p], LV[p], RV[p] = read_factors(fpool, lay, layer, seq, h, int(p))
    theta = float(getattr(cfg, "rope_theta", 0.0))
    if theta > 0:  # keys stored before RoPE: turned at their positions in the oracle too
        return oracle.decode_head_rope(q_rows, kinds, K, V, LK, RK, LV, RV, T, P, theta)
    return oracle.decode_head(q_rows, kinds, K, V, LK, RK, LV, RV, T, P)


def check_page_table(store, cfg, seq: int, layer: int, T: int):
    """Device lengths and page kinds equal the oracle's classification
    (bit-exact); factorized pages point at their own record, dense pages at
    a slot of the dense ring."""
    lay = Layout(cfg)
    assert lengths(store, lay)[seq, layer] == T
    n = (T + cfg.page_size - 1) // cfg.page_size
    kinds, slots = descriptors(store, lay, seq, layer, n)
    ref = oracle.page_kinds(T, cfg.page_size, cfg.sink_tokens, cfg.recent_tokens)
    assert np.array_equal(kinds, ref)
    fac = kinds == oracle.FACTORED
    assert np.array_equal(slots[fac], np.nonzero(fac)[0])
    dense_slots = slots[~fac]
    assert len(set(dense_slots.tolist())) == len(dense_slots)


def spec_of(cfg, inner_rank=12, n_outliers=4, rope_base=None) -> synth.KVSpec:
    return synth.KVSpec(layers=cfg.num_layers, kv_heads=cfg.num_kv_heads, head_dim=cfg.head_dim,
                        page_size=cfg.page_size, inner_rank=inner_rank, n_outliers=n_outliers,
                        rope_base=rope_base, dtype=cfg.kv_dtype)
