"""CPU-side checks of the C-ABI library: it loads, exports every symbol the
header declares, and its host-only logic (page classification, storage
ratio, buffer sizing, argument validation) is right.  No compute calls."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    from page_wise_rank_gb300 import build
    build.build()
    import page_wise_rank_gb300 as m
    return m


def header_functions():
    src = open(os.path.join(ROOT, "include", "puzzlekv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(puzzlekv_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(pkv):
    from page_wise_rank_gb300 import _lib
    declared = header_functions()
    assert declared == sorted(_lib.EXPORTED)
    L = pkv.lib()
    for name in declared:
        assert hasattr(L, name), name


def test_classification_bit_exact_with_oracle(pkv):
    for P in (16, 32, 64):
        for sink, W in ((0, 0), (4, 64), (4, 128), (64, 128), (100, 7)):
            for T in list(range(1, 400)) + [4095, 4096, 4097, 32768, 32769, 131072]:
                a = pkv.classify_pages(T, P, sink, W)
                b = oracle.page_kinds(T, P, sink, W)
                assert a.dtype == np.int32 and np.array_equal(a, b), (T, P, sink, W)


def test_storage_ratio_matches_eq3(pkv):
    for P, d, rk, rv in [(32, 128, 16, 14), (64, 128, 16, 24), (64, 128, 24, 24), (16, 128, 9, 9)]:
        assert pkv.page_storage_ratio(P, d, rk, rv) == oracle.page_storage_ratio(P, d, rk, rv)


def _cfg(pkv, **kw):
    base = dict(num_layers=32, num_kv_heads=8, num_q_heads=32, head_dim=128, page_size=64, rank_k=16, rank_v=24,
                sink_tokens=4, recent_tokens=128, max_batch=1, max_tokens_per_seq=32768 + 256,
                kv_dtype=torch.bfloat16)
    base.update(kw)
    return pkv.StoreConfig(**base)


def test_query_sizes(pkv):
    cfg = _cfg(pkv)
    s = pkv.query_sizes(cfg)
    n_pg = (cfg.max_tokens_per_seq + 63) // 64
    rec = (16 + 24) * (64 + 128) * 2
    assert s["factor_pool"] == 32 * 1 * 8 * n_pg * rec
    dslots = 1 + (128 + 63) // 64 + 2
    assert s["dense_pool"] == 32 * 1 * dslots * 8 * 2 * 64 * 128 * 2
    assert s["workspace"] >= 256 + 32 * 128 * 130 * 4


def test_query_sizes_int4(pkv):
    """INT4 records: 4-bit codes of the four factors plus fp16 scales (r_K + d
    for the key, P + d for the value) -- the Python layout mirror agrees."""
    import oracle
    from store_layout import Layout
    cfg = _cfg(pkv, factor_int4=True)
    s = pkv.query_sizes(cfg)
    n_pg = (cfg.max_tokens_per_seq + 63) // 64
    rec = (16 + 24) * (64 + 128) // 2 + 2 * ((16 + 128) + (64 + 128))
    assert Layout(cfg).rec_bytes == rec
    assert s["factor_pool"] == 32 * 1 * 8 * n_pg * rec
    # the same bytes as the page's storage-ratio accounting (fp16 scales)
    assert rec / (2 * 64 * 128 * 2) == pytest.approx(oracle.int4_page_storage_ratio(64, 128, 16, 24))


@pytest.mark.parametrize("K,N", [(128, 16), (64, 24), (24, 128), (16, 64), (8, 16), (64, 8)])
def test_int4_operand_order_covers_each_element_once(K, N):
    """The INT4 stream order gives every element of a K x N operand exactly one
    (lane, register, element) and fills registers 0 .. K N / 64 - 1 of every lane."""
    from store_layout import _operand_index
    lane, m, e, k, n = _operand_index(K, N)
    assert len(lane) == K * N
    assert len(set(zip(k.tolist(), n.tolist()))) == K * N and k.max() == K - 1 and n.max() == N - 1
    assert len(set(zip(lane.tolist(), m.tolist(), e.tolist()))) == K * N
    assert m.max() == K * N // 64 - 1


@pytest.mark.parametrize("K", [64, 128])
def test_int4_head_dim_scales_in_k_step_order(K):
    """The reader of the head-dim scale vectors (s_RK, s_RV) places column
    16 ks + 8 b + 2 c + e at 16 ks + 4 c + 2 b + e: per 16 columns the four
    lanes c of a row own 4 contiguous halves (the uint2 the decode loads at
    k-step ks), and every column lands once."""
    from store_layout import q4_dscales
    raw = np.arange(K, dtype=np.float16).view(np.uint8)  # stored value = storage position
    got = q4_dscales(raw, K).astype(int)
    want = np.empty(K, dtype=int)
    for ks in range(K // 16):
        for c in range(4):
            for b in range(2):
                for e in range(2):
                    want[16 * ks + 8 * b + 2 * c + e] = 16 * ks + 4 * c + 2 * b + e
    assert np.array_equal(got, want)
    assert sorted(got.tolist()) == list(range(K))


@pytest.mark.parametrize("bad,status", [
    (dict(head_dim=96), 2), (dict(page_size=128), 2), (dict(num_q_heads=33), 1),
    (dict(num_q_heads=8 * 16), 2), (dict(rank_k=0), 1), (dict(rank_v=65), 1),
    (dict(sink_tokens=-1), 1), (dict(max_batch=0), 1),
    (dict(factor_int4=True, kv_dtype=torch.float32), 2), (dict(factor_int4=True, rank_v=40), 2),
    (dict(rope_theta=-1.0), 1), (dict(rope_theta=float("nan")), 1), (dict(rope_theta=1e4, kv_dtype=torch.float32), 2),
    (dict(rope_theta=1e4, factor_int4=True), 2), (dict(rope_theta=1e4, page_size=16, rank_k=8, rank_v=8), 2),
    (dict(rank_k=40, rank_v=40), 2), (dict(rank_k=64, rank_v=64), 2),
])
def test_config_validation(pkv, bad, status):
    with pytest.raises(pkv.PuzzleKVError) as e:
        pkv.query_sizes(_cfg(pkv, **bad))
    assert e.value.status == status
    assert pkv.last_error()


def test_store_create_rejects_bad_pointers_without_gpu(pkv):
    cfg = _cfg(pkv)
    c = cfg.c()
    h = ctypes.c_void_p()
    L = pkv.lib()
    assert L.puzzlekv_store_create(ctypes.byref(c), None, None, None, None, None, ctypes.byref(h)) == 1
    assert L.puzzlekv_store_create(ctypes.byref(c), 16, 256, 256, 256, None, ctypes.byref(h)) == 1  # misaligned
    assert h.value is None
    assert L.puzzlekv_load_prefill(None, 0, None, None, 1, None) == 1
    assert L.puzzlekv_factorize_pages(None, None, None, -1, None) == 1
    assert L.puzzlekv_debug_fail_next_wait(None, 1, 10000) == 1
    assert L.puzzlekv_decode_attention(None, 0, None, None, None, 1, None) == 1
    assert L.puzzlekv_factorize_batch(None, 1, 4, 64, 96, 8, None, None, 0, None, None, None) == 2
    assert L.puzzlekv_factorize_batch(None, 1, 0, 64, 128, 8, None, None, 0, None, None, None) == 0


def test_binding_has_no_cpu_fallback(tmp_path, monkeypatch):
    """Without the built library every call raises instead of computing on the CPU."""
    from page_wise_rank_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.lib()


def test_query_sizes_rope(pkv):
    """Keys before RoPE: the workspace grows by the two fp32 (cos, sin) tables
    (page starts [n_pages][d/2], in-page offsets [P][d/2]); nothing else changes."""
    plain = pkv.query_sizes(_cfg(pkv))
    cfg = _cfg(pkv, rope_theta=5e5)
    rope = pkv.query_sizes(cfg)
    n_pg = (cfg.max_tokens_per_seq + 63) // 64
    assert {k: rope[k] for k in ("dense_pool", "factor_pool", "page_table")} == \
        {k: plain[k] for k in ("dense_pool", "factor_pool", "page_table")}
    extra = rope["workspace"] - plain["workspace"]
    tables = n_pg * 64 * 8 + 64 * 64 * 8
    assert tables <= extra < tables + 512


def test_largest_records_that_fit_decode_shared_memory(pkv):
    """bf16 records of up to 72 padded ranks (K + V) fit the decode kernel's
    8 shared-memory slots at P = 64, d = 128 (28.3 KB each); 80 do not."""
    for rk, rv in ((32, 40), (8, 64), (64, 8)):
        pkv.query_sizes(_cfg(pkv, rank_k=rk, rank_v=rv))
    with pytest.raises(pkv.PuzzleKVError):
        pkv.query_sizes(_cfg(pkv, rank_k=33, rank_v=40))
