"""ctypes binding of libpuzzlekv.so (the C ABI in include/puzzlekv.h).

Argument marshalling only: every step of the hot path runs in the CUDA
library.  There is no CPU fallback -- if the library is missing or fails to
load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpuzzlekv.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_NOT_CONVERGED, ERR_CUDA, ERR_DEVICE_TIMEOUT = range(7)
F32, BF16 = 0, 1
PAGE_FACTORED, PAGE_DENSE = 0, 1

# every symbol include/puzzlekv.h declares
EXPORTED = (
    "puzzlekv_query_sizes",
    "puzzlekv_store_create",
    "puzzlekv_store_destroy",
    "puzzlekv_load_prefill",
    "puzzlekv_factorize_pages",
    "puzzlekv_factorize_layer",
    "puzzlekv_wait_background",
    "puzzlekv_background_stream",
    "puzzlekv_factorize_batch",
    "puzzlekv_int4_record_bytes",
    "puzzlekv_factorize_batch_int4",
    "puzzlekv_append_token",
    "puzzlekv_decode_attention",
    "puzzlekv_decode_step",
    "puzzlekv_convert_ready_pages",
    "puzzlekv_decode_attention_static_scratch",
    "puzzlekv_store_stats",
    "puzzlekv_debug_fail_next_wait",
    "puzzlekv_check_device_status",
    "puzzlekv_factorize_counters",
    "puzzlekv_classify_pages",
    "puzzlekv_page_storage_ratio",
    "puzzlekv_last_error",
)


class PuzzleKVError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"puzzlekv status {status}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "num_kv_heads", "num_q_heads", "head_dim", "page_size", "rank_k", "rank_v",
        "sink_tokens", "recent_tokens", "max_batch", "max_tokens_per_seq", "kv_dtype", "factor_int4")] + [
        ("rope_theta", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with page_wise_rank_gb300.build.build() "
                           "(there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    i32p, i64p, szp = ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(sz)
    cfgp = ctypes.POINTER(Config)
    sig = {
        "puzzlekv_query_sizes": ([cfgp, szp, szp, szp, szp], i32),
        "puzzlekv_store_create": ([cfgp, vp, vp, vp, vp, vp, ctypes.POINTER(vp)], i32),
        "puzzlekv_store_destroy": ([vp], i32),
        "puzzlekv_load_prefill": ([vp, i32, vp, vp, i32, vp], i32),
        "puzzlekv_factorize_pages": ([vp, i32p, i32p, i32, vp], i32),
        "puzzlekv_factorize_layer": ([vp, i32, i32, vp, vp, i32, i32, vp], i32),
        "puzzlekv_wait_background": ([vp, vp], i32),
        "puzzlekv_background_stream": ([vp, ctypes.POINTER(vp)], i32),
        "puzzlekv_factorize_batch": ([vp, i32, i64, i32, i32, i32, vp, vp, i32, vp, vp, vp], i32),
        "puzzlekv_int4_record_bytes": ([i32, i32, i32, i32, i64p], i32),
        "puzzlekv_factorize_batch_int4": ([vp, i64, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp], i32),
        "puzzlekv_append_token": ([vp, i32, vp, vp, i32p, i32, vp], i32),
        "puzzlekv_decode_attention": ([vp, i32, vp, vp, i32p, i32, vp], i32),
        "puzzlekv_decode_attention_static_scratch": ([vp, i32, vp, vp, i32p, i32, vp], i32),
        "puzzlekv_decode_step": ([vp, i32, vp, vp, vp, vp, i32p, i32, vp], i32),
        "puzzlekv_convert_ready_pages": ([vp, vp], i32),
        "puzzlekv_store_stats": ([vp, i32, i32, i32p, i64p, i64p, i64p], i32),
        "puzzlekv_debug_fail_next_wait": ([vp, i32, i64], i32),
        "puzzlekv_check_device_status": ([vp, vp], i32),
        "puzzlekv_factorize_counters": ([vp, vp, i64p, i64p], i32),
        "puzzlekv_classify_pages": ([i32, i32, i32, i32, i32p, i32], i32),
        "puzzlekv_page_storage_ratio": ([i32, i32, i32, i32], ctypes.c_double),
        "puzzlekv_last_error": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def last_error() -> str:
    return lib().puzzlekv_last_error().decode()


def check(status: int) -> None:
    if status != OK:
        raise PuzzleKVError(status, last_error())
