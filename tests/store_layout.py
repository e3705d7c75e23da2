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
        if self.q4:  # INT4 record: key and value code streams, then fp16 scale vectors
            P, d, rkp, rvp = self.P, self.d, self.rkp, self.rvp
            self.q_kslabs = -(-(d * rkp // 64 + rkp * P // 64) // 8)
            self.q_vslabs = -(-(P * rvp // 64 + rvp * d // 64) // 8)
            self.q_off_V = 256 * self.q_kslabs
            self.q_off_sRK = self.q_off_V + 256 * self.q_vslabs
            self.q_off_sRV = self.q_off_sRK + 2 * d
            self.q_off_sLV = self.q_off_sRV + 2 * d
            self.q_off_sLK = self.q_off_sLV + 2 * P
            self.rec_bytes = self.q_off_sLK + 2 * rkp
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


_OPERAND = {}


def _operand_index(K, N):
    """Where each element of a K x N tensor-core B operand sits in a lane's
    register stream: (lane, register, element, k, n) arrays.  Lane l = 4g + c;
    16-wide k-steps (then one 8-wide step if K is an odd multiple of 8), each
    cut into n-tiles of 8, k-step outer; a 16-wide tile gives a lane registers
    (k0 + 2c + e, n0 + g) and (k0 + 8 + 2c + e, n0 + g), an 8-wide tile one."""
    key = (K, N)
    if key not in _OPERAND:
        rows = []
        nt, k16 = N // 8, K // 16
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            for m in range(K * N // 64):
                for e in range(2):
                    if m < k16 * 2 * nt:
                        ks, rem = divmod(m, 2 * nt)
                        k, n = 16 * ks + 8 * (rem & 1) + 2 * c + e, 8 * (rem >> 1) + g
                    else:
                        k, n = 16 * k16 + 2 * c + e, 8 * (m - k16 * 2 * nt) + g
                    rows.append((lane, m, e, k, n))
        _OPERAND[key] = tuple(np.array(col, dtype=np.int64) for col in zip(*rows))
    return _OPERAND[key]


def q4_stream(raw: np.ndarray, nslabs: int) -> np.ndarray:
    """Codes of a stream as [lane][register][element] int: word w of lane l at
    byte ((w // 2) * 32 + l) * 8 + (w % 2) * 4; register m in word m // 4,
    nibbles m % 4 (element 0) and m % 4 + 4 (element 1), each code + 8."""
    words = np.frombuffer(np.asarray(raw, dtype=np.uint8)[: 256 * nslabs].tobytes(), dtype="<u4")
    lane_words = words.reshape(nslabs, 32, 2).transpose(1, 0, 2).reshape(32, 2 * nslabs).astype(np.int64)
    regs = np.empty((32, 8 * nslabs, 2), dtype=np.int64)
    for nu in range(8):
        regs[:, nu % 4::4, nu // 4] = (lane_words >> (4 * nu)) & 15
    return regs - 8


def _operand(codes, m0, K, N):
    lane, m, e, k, n = _operand_index(K, N)
    B = np.empty((K, N), dtype=np.int8)
    B[k, n] = codes[lane, m0 + m, e]
    return B


def q4_scales(raw: np.ndarray, K: int) -> np.ndarray:
    """fp16 scale vector of length K stored in accumulator-column order
    (lane c's elements 8t + 2c, 8t + 2c + 1 contiguous), fp64 in natural order."""
    st = np.frombuffer(np.asarray(raw, dtype=np.uint8)[: 2 * K].tobytes(), dtype=np.float16).astype(np.float64)
    i = np.arange(K)
    return st[((i & 7) >> 1) * (K // 4) + (i >> 3) * 2 + (i & 1)]


def q4_dscales(raw: np.ndarray, K: int) -> np.ndarray:
    """fp16 head-dim scale vector of length K (a multiple of 16) stored in
    k-step order (per 16 columns, lane c's elements 2c, 2c + 1, 8 + 2c,
    9 + 2c contiguous), fp64 in natural order."""
    st = np.frombuffer(np.asarray(raw, dtype=np.uint8)[: 2 * K].tobytes(), dtype=np.float16).astype(np.float64)
    n = np.arange(K)
    return st[(n >> 4) * 16 + ((n & 7) >> 1) * 4 + ((n >> 3) & 1) * 2 + (n & 1)]


def read_record_q4(rec: np.ndarray, lay: Layout):
    """INT4 record -> codes and fp16 scales of each factor, as a dict
    {name: (codes [rows][cols] int8, scales fp64, per_row)} in the orientation
    LK [P][rkp], RK [rkp][d], LVt [rvp][P], RVt [d][rvp], plus "pad": the codes
    of the streams' unused registers."""
    P, d, rkp, rvp = lay.P, lay.d, lay.rkp, lay.rvp
    ks = q4_stream(rec, lay.q_kslabs)
    vs = q4_stream(rec[lay.q_off_V:], lay.q_vslabs)
    nk, nv = d * rkp // 64, P * rvp // 64
    RK_B, LK_B = _operand(ks, 0, d, rkp), _operand(ks, nk, rkp, P)  # B[head dim][rank], B[rank][token]
    LV_B, RV_B = _operand(vs, 0, P, rvp), _operand(vs, nv, rvp, d)  # B[token][rank], B[rank][head dim]
    pad = np.concatenate([ks[:, nk + rkp * P // 64:].ravel(), vs[:, nv + rvp * d // 64:].ravel()])
    return {"LK": (LK_B.T, q4_scales(rec[lay.q_off_sLK:], rkp), False),
            "RK": (RK_B.T, q4_dscales(rec[lay.q_off_sRK:], d), False),
            "LVt": (LV_B.T, q4_scales(rec[lay.q_off_sLV:], P), False),
            "RVt": (RV_B.T, q4_dscales(rec[lay.q_off_sRV:], d), True),
            "pad": pad}


def read_record(rec: np.ndarray, lay: Layout):
    """Factors of one record given its rec_bytes bytes, fp64 (INT4 records dequantized exactly)."""
    if lay.q4:
        q = read_record_q4(rec, lay)
        q.pop("pad")
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
