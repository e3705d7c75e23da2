"""Test-side reader of the store's documented device layout (include/puzzlekv.h,
csrc/layout.h): page-table entries and factor records, unpacked from raw
bytes copied back to the host.  Used to hand the GPU's stored factors and
page descriptors to the oracle; it re-derives offsets from the documented
format instead of calling the library.
"""
from __future__ import annotations

from math import gcd

import numpy as np
import torch

KIND_SHIFT = 30
MAX_SPLITS = 128


def _r8(x):
    return (x + 7) // 8 * 8


class Layout:
    def __init__(self, cfg):
        self.L, self.H, self.Hq = cfg.num_layers, cfg.num_kv_heads, cfg.num_q_heads
        self.d, self.P = cfg.head_dim, cfg.page_size
        self.rk, self.rv = cfg.rank_k, cfg.rank_v
        self.rkp, self.rvp = _r8(cfg.rank_k), _r8(cfg.rank_v)
        self.Bmax, self.Tmax = cfg.max_batch, cfg.max_tokens_per_seq
        self.esz = 2 if cfg.kv_dtype == torch.bfloat16 else 4
        self.dtype = cfg.kv_dtype
        self.n_pg_max = (self.Tmax + self.P - 1) // self.P
        e = self.esz
        self.off_RK = self.P * self.rkp * e
        self.off_LV = self.off_RK + self.rkp * self.d * e
        self.off_RV = self.off_LV + self.rvp * self.P * e
        self.rec_bytes = self.off_RV + self.d * self.rvp * e
        self.q4 = bool(getattr(cfg, "factor_int4", False))
        if self.q4:  # INT4 record: code blocks, then fp16 scale blocks
            P, d, rkp, rvp = self.P, self.d, self.rkp, self.rvp
            self.q_off_RK = P * rkp // 2
            self.q_off_LV = self.q_off_RK + rkp * d // 2
            self.q_off_RV = self.q_off_LV + rvp * P // 2
            self.q_off_sLK = self.q_off_RV + d * rvp // 2
            self.q_off_sRK = self.q_off_sLK + 2 * rkp
            self.q_off_sLV = self.q_off_sRK + 2 * d
            self.q_off_sRV = self.q_off_sLV + 2 * P
            self.rec_bytes = self.q_off_sRV + 2 * d
        self.desc_offset = (self.Bmax * self.L * 4 + 255) // 256 * 256

    def record_offset(self, l, b, h, p):
        return (((l * self.Bmax + b) * self.H + h) * self.n_pg_max + p) * self.rec_bytes


def swizzle_chunk(row, c, C):
    g = gcd(C, 8)
    if g == 1:
        return c
    return c ^ ((row // (8 // g)) & (g - 1))


_PERM = {}


def _perm(rows, C):
    key = (rows, C)
    if key not in _PERM:
        _PERM[key] = np.array([[swizzle_chunk(r, c, C) for c in range(C)] for r in range(rows)], dtype=np.int64)
    return _PERM[key]


def unswizzle(raw: np.ndarray, rows: int, cols: int, esz: int, dtype) -> np.ndarray:
    """Rows of `cols` elements stored with the 16-byte chunk XOR swizzle -> [rows, cols] fp64."""
    C = cols * esz // 16
    chunks = raw.reshape(rows, C, 16)
    out = chunks[np.arange(rows)[:, None], _perm(rows, C)]
    t = torch.from_numpy(np.ascontiguousarray(out).reshape(-1)).view(dtype).reshape(rows, cols)
    return t.double().numpy()


def lengths(store, lay: Layout) -> np.ndarray:
    pt = store.page_table.cpu().numpy()
    return pt[: lay.Bmax * lay.L * 4].view(np.int32).reshape(lay.Bmax, lay.L).copy()


def descriptors(store, lay: Layout, b: int, l: int, n_pages: int):
    pt = store.page_table.cpu().numpy()
    desc = pt[lay.desc_offset:].view(np.int32)[: lay.Bmax * lay.L * lay.n_pg_max].reshape(lay.Bmax, lay.L, lay.n_pg_max)
    d = desc[b, l, :n_pages]
    return (d >> KIND_SHIFT).astype(np.int32), (d & ((1 << KIND_SHIFT) - 1)).astype(np.int32)


def read_factors(fp_bytes: np.ndarray, lay: Layout, l: int, b: int, h: int, p: int):
    """(LK [P, rk], RK [rk, d], LV [P, rv], RV [rv, d]) of one record, fp64."""
    o = lay.record_offset(l, b, h, p)
    return read_record(fp_bytes[o:o + lay.rec_bytes], lay)


def q4_codes(raw: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Signed INT4 codes of a row-major [rows][cols] block (code + 8, low nibble first)."""
    b = np.asarray(raw, dtype=np.uint8)[: rows * cols // 2]
    n = np.empty(rows * cols, dtype=np.int16)
    n[0::2] = b & 15
    n[1::2] = b >> 4
    return (n - 8).reshape(rows, cols).astype(np.int8)


def read_record_q4(rec: np.ndarray, lay: Layout):
    """INT4 record -> codes and fp16 scales of each factor, as a dict
    {name: (codes [rows][cols] int8, scales fp64, per_row)} in the record orientation."""
    P, d, rkp, rvp = lay.P, lay.d, lay.rkp, lay.rvp
    sc = lambda off, n: np.frombuffer(rec[off:off + 2 * n].tobytes(), dtype=np.float16).astype(np.float64)
    return {"LK": (q4_codes(rec[:], P, rkp), sc(lay.q_off_sLK, rkp), False),
            "RK": (q4_codes(rec[lay.q_off_RK:], rkp, d), sc(lay.q_off_sRK, d), False),
            "LVt": (q4_codes(rec[lay.q_off_LV:], rvp, P), sc(lay.q_off_sLV, P), False),
            "RVt": (q4_codes(rec[lay.q_off_RV:], d, rvp), sc(lay.q_off_sRV, d), True)}


def read_record(rec: np.ndarray, lay: Layout):
    """Factors of one record given its rec_bytes bytes, fp64 (INT4 records dequantized exactly)."""
    if lay.q4:
        q = read_record_q4(rec, lay)
        deq = {k: c.astype(np.float64) * (s[:, None] if per_row else s[None, :]) for k, (c, s, per_row) in q.items()}
        return (deq["LK"][:, : lay.rk], deq["RK"][: lay.rk], deq["LVt"][: lay.rv].T.copy(),
                deq["RVt"][:, : lay.rv].T.copy())
    e, P, d = lay.esz, lay.P, lay.d
    LK = unswizzle(rec[: lay.off_RK], P, lay.rkp, e, lay.dtype)[:, : lay.rk]
    RK = unswizzle(rec[lay.off_RK: lay.off_LV], lay.rkp, d, e, lay.dtype)[: lay.rk]
    LVt = unswizzle(rec[lay.off_LV: lay.off_RV], lay.rvp, P, e, lay.dtype)[: lay.rv]
    RVt = unswizzle(rec[lay.off_RV: lay.rec_bytes], d, lay.rvp, e, lay.dtype)[:, : lay.rv]
    return LK, RK, LVt.T.copy(), RVt.T.copy()


def factor_pool_slice(store, lay: Layout, l: int, b: int, h: int) -> np.ndarray:
    """Host copy of the records of one (layer, seq, head), indexed from byte 0 of the pool
    (other bytes left zero) -- avoids copying the whole pool for large configs."""
    o0 = lay.record_offset(l, b, h, 0)
    n = lay.n_pg_max * lay.rec_bytes
    buf = np.zeros(o0 + n, dtype=np.uint8)
    buf[o0:o0 + n] = store.factor_pool[o0:o0 + n].cpu().numpy()
    return buf
