"""PuzzleKV page-wise low-rank KV cache compression on GB300 (sm_103a).

Python face of the C ABI in include/puzzlekv.h.  The functions here only
marshal arguments (shapes, dtypes, pointers, the current CUDA stream) into
the CUDA library; PyTorch provides device memory and streams.  Citations name
sections/equations of "PuzzleKV: Page-Wise Low-Rank Decomposition for KV
Cache Compression".
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import _lib
from ._lib import BF16, F32, PAGE_DENSE, PAGE_FACTORED, PuzzleKVError, check, last_error, lib  # noqa: F401

_DT = {torch.float32: F32, torch.bfloat16: BF16}
_TORCH = {F32: torch.float32, BF16: torch.bfloat16}


@dataclass(frozen=True)
class StoreConfig:
    num_layers: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    page_size: int
    rank_k: int
    rank_v: int
    sink_tokens: int
    recent_tokens: int
    max_batch: int
    max_tokens_per_seq: int
    kv_dtype: torch.dtype = torch.bfloat16
    factor_int4: bool = False
    rope_theta: float = 0.0  # > 0: keys are given before RoPE with this base and turned at attention

    def c(self) -> _lib.Config:
        c = _lib.Config()
        for name, ctype in _lib.Config._fields_:
            if name == "kv_dtype":
                setattr(c, name, _DT[self.kv_dtype])
            elif ctype is ctypes.c_float:
                setattr(c, name, float(getattr(self, name)))
            else:
                setattr(c, name, int(getattr(self, name)))
        return c


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, shape, dtype, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


_SEQ_CACHE: dict = {}


def _seq_ids(seq_ids: Sequence[int]):
    key = tuple(int(s) for s in seq_ids)
    arr = _SEQ_CACHE.get(key)
    if arr is None:
        if len(_SEQ_CACHE) > 4096:
            _SEQ_CACHE.clear()
        arr = _SEQ_CACHE[key] = (ctypes.c_int32 * len(key))(*key)
    return arr, len(key)


def query_sizes(cfg: StoreConfig) -> dict:
    """Byte sizes of the dense pool, factor pool, page table and workspace."""
    s = [ctypes.c_size_t() for _ in range(4)]
    c = cfg.c()
    check(lib().puzzlekv_query_sizes(ctypes.byref(c), *[ctypes.byref(x) for x in s]))
    return dict(zip(("dense_pool", "factor_pool", "page_table", "workspace"), (x.value for x in s)))


def classify_pages(T: int, P: int, sink_tokens: int, recent_tokens: int) -> np.ndarray:
    """PAGE_DENSE / PAGE_FACTORED per page of a T-token sequence (host-only)."""
    n = (T + P - 1) // P
    out = (ctypes.c_int32 * max(n, 1))()
    got = lib().puzzlekv_classify_pages(T, P, sink_tokens, recent_tokens, out, n)
    if got != n:
        raise ValueError("bad arguments to classify_pages")
    return np.frombuffer(out, dtype=np.int32, count=n).copy()


def page_storage_ratio(P: int, d: int, rank_k: int, rank_v: int) -> float:
    """(r_K + r_V)(P + d) / (2 P d), eq. (3)."""
    return float(lib().puzzlekv_page_storage_ratio(P, d, rank_k, rank_v))


def factorize_batch(X: torch.Tensor, r: int, out_dtype: torch.dtype = torch.float32, sigma: bool = True,
                    stream: Optional[torch.cuda.Stream] = None):
    """Factorize independent pages X[n, P, d] -> (L[n, P, r], R[n, r, d], sigma[n, P] or None, status[1]).

    ``status`` (int32 on the device) is nonzero if an eigensolve hit its iteration cap.
    """
    if X.dim() != 3:
        raise ValueError("X must be [n, P, d]")
    n, P, d = X.shape
    _need(X, (n, P, d), X.dtype, "X")
    if X.dtype not in _DT:
        raise ValueError("X must be float32 or bfloat16")
    L = torch.empty(n, P, r, dtype=out_dtype, device=X.device)
    R = torch.empty(n, r, d, dtype=out_dtype, device=X.device)
    S = torch.empty(n, P, dtype=torch.float32, device=X.device) if sigma else None
    status = torch.zeros(1, dtype=torch.int32, device=X.device)
    check(lib().puzzlekv_factorize_batch(_ptr(X), _DT[X.dtype], n, P, d, r, _ptr(L), _ptr(R), _DT[out_dtype],
                                         _ptr(S) if S is not None else None, _ptr(status), _stream(stream)))
    return L, R, S, status


def int4_record_bytes(P: int, d: int, rank_k: int, rank_v: int) -> int:
    """Bytes of one INT4 factor record (§4.3) of a store with these shapes."""
    b = ctypes.c_int64()
    check(lib().puzzlekv_int4_record_bytes(P, d, rank_k, rank_v, ctypes.byref(b)))
    return b.value


def factorize_batch_int4(X: torch.Tensor, rank_k: int, rank_v: int, kind: int, absorbed: bool = True,
                         stream: Optional[torch.cuda.Stream] = None):
    """INT4 records of independent bf16 pages X[n, P, d] (§4.3): returns (records uint8
    [n, record_bytes], L~ fp32 [n, P, rp] or None, R~ fp32 [n, rp, d] or None, status[1]);
    kind 0 = key pages at rank_k, 1 = value pages at rank_v."""
    if X.dim() != 3 or X.dtype != torch.bfloat16:
        raise ValueError("X must be bf16 [n, P, d]")
    n, P, d = X.shape
    _need(X, (n, P, d), torch.bfloat16, "X")
    rb = int4_record_bytes(P, d, rank_k, rank_v)
    rp = ((rank_k if kind == 0 else rank_v) + 7) // 8 * 8
    rec = torch.zeros(n, rb, dtype=torch.uint8, device=X.device)
    Lq = torch.empty(n, P, rp, dtype=torch.float32, device=X.device) if absorbed else None
    Rq = torch.empty(n, rp, d, dtype=torch.float32, device=X.device) if absorbed else None
    status = torch.zeros(1, dtype=torch.int32, device=X.device)
    check(lib().puzzlekv_factorize_batch_int4(_ptr(X), n, P, d, rank_k, rank_v, kind, _ptr(rec),
                                              _ptr(Lq) if absorbed else None, _ptr(Rq) if absorbed else None,
                                              _ptr(status), _stream(stream)))
    return rec, Lq, Rq, status


class Store:
    """Paged factor store over four torch-allocated device buffers."""

    def __init__(self, cfg: StoreConfig, device="cuda", stream: Optional[torch.cuda.Stream] = None):
        self.cfg = cfg
        sizes = query_sizes(cfg)
        self.sizes = sizes
        # 256-byte aligned device buffers (the caching allocator aligns to 512)
        self.dense_pool = torch.empty(sizes["dense_pool"], dtype=torch.uint8, device=device)
        self.factor_pool = torch.empty(sizes["factor_pool"], dtype=torch.uint8, device=device)
        self.page_table = torch.empty(sizes["page_table"], dtype=torch.uint8, device=device)
        self.workspace = torch.empty(sizes["workspace"], dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        c = cfg.c()
        check(lib().puzzlekv_store_create(ctypes.byref(c), _ptr(self.dense_pool), _ptr(self.factor_pool),
                                          _ptr(self.page_table), _ptr(self.workspace), _stream(stream),
                                          ctypes.byref(h)))
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().puzzlekv_store_destroy(self._h)  # waits for the background stream
            self._h = None
            self._inputs = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def load_prefill(self, seq: int, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        """Prefill compression of sequence `seq` from dense k, v [L, H, T, d] (§3.3 ①②③)."""
        c = self.cfg
        T = k.shape[2]
        shape = (c.num_layers, c.num_kv_heads, T, c.head_dim)
        _need(k, shape, c.kv_dtype, "k")
        _need(v, shape, c.kv_dtype, "v")
        check(lib().puzzlekv_load_prefill(self._h, seq, _ptr(k), _ptr(v), T, _stream(stream)))

    def factorize_pages(self, pages: Optional[Sequence[tuple]] = None, stream=None) -> None:
        """Factorize the listed completed pages [(seq, page), ...] of every layer, or
        every eligible page when `pages` is None (§3.3 ③⑤); pages with factors are skipped."""
        if pages is None:
            check(lib().puzzlekv_factorize_pages(self._h, None, None, -1, _stream(stream)))
            return
        n = len(pages)
        seqs = (ctypes.c_int32 * max(n, 1))(*[int(b) for b, _ in pages])
        pgs = (ctypes.c_int32 * max(n, 1))(*[int(p) for _, p in pages])
        check(lib().puzzlekv_factorize_pages(self._h, seqs, pgs, n, _stream(stream)))

    def factorize_layer(self, seq: int, layer: int, k: torch.Tensor, v: torch.Tensor, background: bool = True,
                        stream=None) -> None:
        """Prefill compression of one layer from dense k, v [H, T, d] (§3.3 ①②③).  With
        `background`, the factorization runs on the store's internal stream so that the
        caller's later layers overlap it; the store then keeps k and v referenced until
        that stream is past the call (or until wait_background / close)."""
        c = self.cfg
        T = k.shape[1]
        shape = (c.num_kv_heads, T, c.head_dim)
        _need(k, shape, c.kv_dtype, "k")
        _need(v, shape, c.kv_dtype, "v")
        self._release_inputs()
        check(lib().puzzlekv_factorize_layer(self._h, seq, layer, _ptr(k), _ptr(v), T, int(background),
                                             _stream(stream)))
        if background:  # k and v stay referenced until the background stream is past this call
            ev = torch.cuda.Event()
            ev.record(self.background_stream())
            self._inputs.append((ev, k, v))

    def _release_inputs(self) -> None:
        """Drop the references to background prefill inputs the internal stream is done with."""
        inputs = getattr(self, "_inputs", None)
        if inputs is None:
            self._inputs = []
            return
        while inputs and inputs[0][0].query():
            inputs.pop(0)

    def wait_background(self, stream=None) -> None:
        """Order `stream` after all background work queued so far (conversions, layer prefills)."""
        check(lib().puzzlekv_wait_background(self._h, _stream(stream)))
        self._release_inputs()

    def background_stream(self) -> torch.cuda.ExternalStream:
        """The store's internal low-priority stream, as a torch stream object."""
        if getattr(self, "_bg", None) is None:
            h = ctypes.c_void_p()
            check(lib().puzzlekv_background_stream(self._h, ctypes.byref(h)))
            self._bg = torch.cuda.ExternalStream(h.value, device=self.dense_pool.device)
        return self._bg

    def append_token(self, layer: int, k: torch.Tensor, v: torch.Tensor, seq_ids: Sequence[int], stream=None) -> None:
        """Append one token per sequence to `layer`; converts pages leaving the window (§3.3 ⑤)."""
        c = self.cfg
        ids, B = _seq_ids(seq_ids)
        _need(k, (B, c.num_kv_heads, c.head_dim), c.kv_dtype, "k")
        _need(v, (B, c.num_kv_heads, c.head_dim), c.kv_dtype, "v")
        check(lib().puzzlekv_append_token(self._h, layer, _ptr(k), _ptr(v), ids, B, _stream(stream)))

    def decode_attention(self, layer: int, q: torch.Tensor, out: torch.Tensor, seq_ids: Sequence[int],
                         stream=None) -> torch.Tensor:
        """Mixed dense/factorized decode attention of one layer (§3.3 ④, eqs. (4)-(5))."""
        c = self.cfg
        ids, B = _seq_ids(seq_ids)
        _need(q, (B, c.num_q_heads, c.head_dim), c.kv_dtype, "q")
        _need(out, (B, c.num_q_heads, c.head_dim), torch.float32, "out")
        check(lib().puzzlekv_decode_attention(self._h, layer, _ptr(q), _ptr(out), ids, B, _stream(stream)))
        return out

    def decode_step(self, layer: int, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                    seq_ids: Sequence[int], stream=None) -> torch.Tensor:
        """Append (k, v) and attend with q in one launch (§3.3 ④⑤); converts the
        page leaving the window first."""
        c = self.cfg
        ids, B = _seq_ids(seq_ids)
        _need(q, (B, c.num_q_heads, c.head_dim), c.kv_dtype, "q")
        _need(k, (B, c.num_kv_heads, c.head_dim), c.kv_dtype, "k")
        _need(v, (B, c.num_kv_heads, c.head_dim), c.kv_dtype, "v")
        _need(out, (B, c.num_q_heads, c.head_dim), torch.float32, "out")
        check(lib().puzzlekv_decode_step(self._h, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(out), ids, B,
                                         _stream(stream)))
        return out

    def convert_ready_pages(self, stream=None) -> None:
        """Factorize every complete, not yet factorized page of all sequences and
        layers in one batched launch (ahead of its leaving the window)."""
        check(lib().puzzlekv_convert_ready_pages(self._h, _stream(stream)))

    def decode_attention_static_scratch(self, layer: int, q: torch.Tensor, out: torch.Tensor,
                                        seq_ids: Sequence[int], stream=None) -> torch.Tensor:
        """decode_attention with its split-K scratch in the library's static
        device array (no per-call scratch buffer; see include/puzzlekv.h)."""
        c = self.cfg
        ids, B = _seq_ids(seq_ids)
        _need(q, (B, c.num_q_heads, c.head_dim), c.kv_dtype, "q")
        _need(out, (B, c.num_q_heads, c.head_dim), torch.float32, "out")
        check(lib().puzzlekv_decode_attention_static_scratch(self._h, layer, _ptr(q), _ptr(out), ids, B,
                                                             _stream(stream)))
        return out

    def stats(self, seq: int, layer: int) -> dict:
        n = ctypes.c_int32()
        nd, nf, nb = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check(lib().puzzlekv_store_stats(self._h, seq, layer, ctypes.byref(n), ctypes.byref(nd), ctypes.byref(nf),
                                         ctypes.byref(nb)))
        return {"length": n.value, "dense_pages": nd.value, "factored_pages": nf.value, "bytes_live": nb.value}

    def debug_fail_next_wait(self, where: int, wait_ns: int = 100_000) -> None:
        """Test hook of the failure path: the next decode launch's wait at `where`
        (1 = a unit copy, 2 = the split merge) runs out after wait_ns (see include/puzzlekv.h)."""
        check(lib().puzzlekv_debug_fail_next_wait(self._h, int(where), int(wait_ns)))

    def check_device_status(self, stream=None) -> int:
        """Synchronise and return the status code (raises nothing; OK = 0)."""
        st = lib().puzzlekv_check_device_status(self._h, _stream(stream))
        self._release_inputs()
        return st

    def factorize_counters(self, stream=None) -> tuple:
        """(page jobs, QL rotations) of the store's factorization launches since
        the last call (rotations come only from jobs of rank above P / 2);
        the counters are cleared."""
        jobs, rotations = ctypes.c_int64(0), ctypes.c_int64(0)
        check(lib().puzzlekv_factorize_counters(self._h, _stream(stream), ctypes.byref(jobs), ctypes.byref(rotations)))
        return jobs.value, rotations.value
