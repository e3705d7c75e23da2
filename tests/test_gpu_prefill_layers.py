"""Layer-by-layer prefill compression [PuzzleKV §3.3 ①②③, §4.5 time to first token].

puzzlekv_factorize_layer runs the same kernels as the whole-prompt
puzzlekv_factorize_pages, restricted to one layer; in the background form the
factorization runs on the store's internal stream while the caller's stream
goes on.  Both must leave the store byte for byte as the whole-prompt call
does (the factorization and the page-table writes are deterministic), and
decode on either store must give bitwise equal outputs -- whether or not the
caller waits for the background work first, since decode waits for it.
"""
import pytest
import torch

import synth
from gpu_helpers import spec_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from page_wise_rank_gb300 import build
    build.build()
    import page_wise_rank_gb300 as m
    return m


def cfg_of(pkv, **kw):
    base = dict(num_layers=4, num_kv_heads=2, num_q_heads=8, head_dim=128, page_size=64, rank_k=16, rank_v=24,
                sink_tokens=4, recent_tokens=128, max_batch=2, max_tokens_per_seq=4200, kv_dtype=torch.bfloat16)
    base.update(kw)
    return pkv.StoreConfig(**base)


def fresh(pkv, cfg):
    st = pkv.Store(cfg)
    st.dense_pool.zero_()  # pages no call writes stay equal between stores
    st.factor_pool.zero_()
    return st


def state(store):
    torch.cuda.synchronize()
    return [t.clone() for t in (store.dense_pool, store.factor_pool, store.page_table)]


@pytest.mark.parametrize("int4", [False, True])
def test_layer_prefill_matches_whole_prompt(pkv, int4):
    cfg = cfg_of(pkv, factor_int4=int4)
    T = 3000
    K, V = synth.prefill_kv(spec_of(cfg), T, seq=1, device="cuda")
    ref = fresh(pkv, cfg)
    ref.factorize_pages(1, K, V)
    want = state(ref)
    for background in (False, True):
        st = fresh(pkv, cfg)
        for l in range(cfg.num_layers):
            k, v = K[l].clone(), V[l].clone()
            st.factorize_layer(1, l, k, v, background=background)
            del k, v
            # the caller's stream moves on at once: fresh allocations (which
            # must not take k / v's memory while the background still reads it)
            junk = torch.full((cfg.num_kv_heads, T, cfg.head_dim), float("nan"), dtype=torch.bfloat16,
                              device="cuda")
            del junk
        st.wait_background()
        got = state(st)
        for a, b, name in zip(want, got, ("dense pool", "factor pool", "page table")):
            assert torch.equal(a, b), (name, background)
        assert st.check_device_status() == 0


def test_decode_waits_for_background_prefill(pkv):
    cfg = cfg_of(pkv)
    T = 4000
    K, V = synth.prefill_kv(spec_of(cfg), T, seq=0, device="cuda")
    ref = pkv.Store(cfg)
    ref.factorize_pages(0, K, V)
    st = pkv.Store(cfg)
    for l in range(cfg.num_layers):
        st.factorize_layer(0, l, K[l].clone(), V[l].clone(), background=True)
    # no wait: the decode calls order themselves after the background work
    q = synth.queries(1, cfg.num_q_heads, cfg.head_dim, step=3, layer=2).cuda()
    for l in range(cfg.num_layers):
        a = torch.empty(1, cfg.num_q_heads, cfg.head_dim, device="cuda")
        b = torch.empty_like(a)
        ref.decode_attention(l, q, a, [0])
        st.decode_attention(l, q, b, [0])
        assert torch.equal(a, b), l
    assert st.check_device_status() == 0


def test_layer_prefill_validation(pkv):
    cfg = cfg_of(pkv)
    st = pkv.Store(cfg)
    k = torch.zeros(cfg.num_kv_heads, 100, cfg.head_dim, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PuzzleKVError):
        pkv.check(pkv.lib().puzzlekv_factorize_layer(st.handle, 0, cfg.num_layers, pkv._ptr(k), pkv._ptr(k), 100,
                                                     1, pkv._stream(None)))
    with pytest.raises(pkv.PuzzleKVError):
        pkv.check(pkv.lib().puzzlekv_factorize_layer(st.handle, 5, 0, pkv._ptr(k), pkv._ptr(k), 100, 1,
                                                     pkv._stream(None)))
