"""The C-ABI boundary calls of prefill and page-list factorization
[PuzzleKV §3.3 ③ and ⑤]: puzzlekv_load_prefill (a sequence's dense prompt
cache in, its eligible pages factorized) and puzzlekv_factorize_pages (a
caller-chosen list of completed pages, or every eligible page with n = -1).

A listed page inside the local window gets its factor records at once but
stays dense for attention until it leaves the window; the step that moves it
out then only switches it to those factors.  The records equal the stateless
factorization of the same page rows (same kernel), decode is compared with
the oracle on the stored factors (2e-3 per output row), page tables
bit-exactly, and a bad entry changes nothing.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import HostCache, check_page_table, oracle_decode_on_store, rel_err_rows, spec_of
from store_layout import Layout, read_factors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from page_wise_rank_gb300 import build
    build.build()
    import page_wise_rank_gb300 as m
    return m


def make(pkv, T=3000, W=512):
    cfg = pkv.StoreConfig(num_layers=2, num_kv_heads=2, num_q_heads=8, head_dim=128, page_size=64, rank_k=16,
                          rank_v=24, sink_tokens=4, recent_tokens=W, max_batch=2, max_tokens_per_seq=4096,
                          kv_dtype=torch.bfloat16)
    spec = spec_of(cfg, rope_base=5e5)
    store = pkv.Store(cfg)
    store.factor_pool.zero_()
    host = HostCache()
    K, V = synth.prefill_kv(spec, T, seq=0)
    store.load_prefill(0, K.cuda(), V.cuda())
    host.set_prefill(0, K, V)
    return cfg, spec, store, host


def decode_all(store, cfg, layer, step):
    q = synth.queries(1, cfg.num_q_heads, cfg.head_dim, step=step, layer=layer)
    out = torch.empty(1, cfg.num_q_heads, cfg.head_dim, device="cuda")
    store.decode_attention(layer, q.cuda(), out, [0])
    return q, out


def records_match_stateless(pkv, store, cfg, host, pages):
    """The records of the listed pages (every layer and KV head) equal the
    stateless factorization of the page rows, rounded to bf16."""
    lay, P = Layout(cfg), cfg.page_size
    fpool = store.factor_pool.cpu().numpy()
    for l in range(cfg.num_layers):
        for kind, r in ((0, cfg.rank_k), (1, cfg.rank_v)):
            rows = [host.rows(0, l, h)[kind] for h in range(cfg.num_kv_heads)]
            X = torch.tensor(np.stack([rows[h][p * P:(p + 1) * P] for h in range(cfg.num_kv_heads) for p in pages]),
                             dtype=torch.bfloat16, device="cuda")
            L_, R_, _, st = pkv.factorize_batch(X, r, out_dtype=torch.bfloat16, sigma=False)
            L_, R_ = L_.double().cpu().numpy(), R_.double().cpu().numpy()
            i = 0
            for h in range(cfg.num_kv_heads):
                for p in pages:
                    f = read_factors(fpool, lay, l, 0, h, p)
                    got = (f[0], f[1]) if kind == 0 else (f[2], f[3])
                    assert np.array_equal(got[0], L_[i]) and np.array_equal(got[1], R_[i]), (l, kind, h, p)
                    i += 1


def test_listed_window_pages_switch_to_their_factors(pkv):
    cfg, spec, store, host = make(pkv)
    P, W, T = cfg.page_size, cfg.recent_tokens, 3000
    kinds = oracle.page_kinds(T, P, cfg.sink_tokens, W)
    window = [p for p in range(T // P) if kinds[p] == oracle.DENSE and p > 0]  # complete dense pages
    assert window == list(range(38, 46))
    q0, before = decode_all(store, cfg, 1, step=0)
    store.factorize_pages([(0, 40), (0, 42), (0, 40)])
    records_match_stateless(pkv, store, cfg, host, [40, 42])
    # still dense for attention: the same output, bit for bit
    _, after = decode_all(store, cfg, 1, step=0)
    assert torch.equal(before, after)
    for l in range(cfg.num_layers):
        check_page_table(store, cfg, 0, l, T)
    # grow until page 42 has left the window: its factors are used
    T1 = (42 + 1) * P + W
    steps = T1 - T
    cache = {}
    for s in range(steps):
        for l in range(cfg.num_layers):
            k, v = synth.decode_tokens(spec, l, [0], [T + s], device="cuda", cache=cache)
            q = synth.queries(1, cfg.num_q_heads, cfg.head_dim, step=s, layer=l).cuda()
            out = torch.empty(1, cfg.num_q_heads, cfg.head_dim, device="cuda")
            store.decode_step(l, q, k, v, out, [0])
            host.append(0, l, k[0], v[0])
    assert store.check_device_status() == 0, pkv.last_error()
    records_match_stateless(pkv, store, cfg, host, [40, 42])  # never refactorized
    G = cfg.num_q_heads // cfg.num_kv_heads
    for l in range(cfg.num_layers):
        check_page_table(store, cfg, 0, l, T1)
        q, out = decode_all(store, cfg, l, step=7)
        assert store.check_device_status() == 0
        got = out.cpu().double().numpy()[0]
        for h in range(cfg.num_kv_heads):
            ref = oracle_decode_on_store(store, cfg, host, 0, l, h, q[0, h * G:(h + 1) * G].double().numpy())
            assert rel_err_rows(got[h * G:(h + 1) * G], ref) <= 2e-3


def test_all_eligible_pages(pkv):
    cfg, spec, store, host = make(pkv)
    store.factorize_pages(None)
    records_match_stateless(pkv, store, cfg, host, list(range(38, 46)))
    before = store.factor_pool.clone()
    store.factorize_pages(None)  # nothing left to do
    store.factorize_pages([(0, 39)])  # already factorized: skipped
    assert torch.equal(before, store.factor_pool)
    assert store.check_device_status() == 0


@pytest.mark.parametrize("bad", [(0, 0), (0, 46), (0, 100), (0, -1), (1, 40), (2, 40), (-1, 40)])
def test_bad_entry_changes_nothing(pkv, bad):
    """A list with one bad entry (sink page, incomplete page, page out of
    range, empty or out-of-range sequence slot) is refused as a whole."""
    cfg, spec, store, host = make(pkv)
    torch.cuda.synchronize()
    before = store.factor_pool.clone()
    with pytest.raises(pkv.PuzzleKVError) as e:
        store.factorize_pages([(0, 41), bad])
    assert e.value.status == pkv._lib.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(before, store.factor_pool)
    store.factorize_pages([(0, 41)])  # the good entry alone: not marked by the refused call
    records_match_stateless(pkv, store, cfg, host, [41])
    assert store.check_device_status() == 0


def test_load_prefill_against_oracle(pkv):
    cfg, spec, store, host = make(pkv, T=2345, W=128)
    G = cfg.num_q_heads // cfg.num_kv_heads
    for l in range(cfg.num_layers):
        check_page_table(store, cfg, 0, l, 2345)
        q, out = decode_all(store, cfg, l, step=2)
        assert store.check_device_status() == 0
        got = out.cpu().double().numpy()[0]
        for h in range(cfg.num_kv_heads):
            ref = oracle_decode_on_store(store, cfg, host, 0, l, h, q[0, h * G:(h + 1) * G].double().numpy())
            assert rel_err_rows(got[h * G:(h + 1) * G], ref) <= 2e-3
