"""Keys stored before RoPE [PuzzleKV §4.1, Appendix D.3] on the GPU.

The store factorizes unrotated keys and turns every key -- reconstructed from
its page's factors or read from a dense page -- by RoPE at its absolute
position inside the decode kernel.  The oracle does the same in fp64 on the
factors the store holds (decode_head_rope: reconstruct, rotate, plain
softmax); the GPU must agree within the bf16 bar, 2e-3 per row (decode on
identical factors).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import HostCache, check_page_table, oracle_decode_on_store, rel_err_rows, spec_of

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from page_wise_rank_gb300 import build
    build.build()
    import page_wise_rank_gb300 as m
    return m


def cfg_rope(pkv, **kw):
    base = dict(num_layers=2, num_kv_heads=2, num_q_heads=8, head_dim=128, page_size=64, rank_k=16, rank_v=24,
                sink_tokens=4, recent_tokens=128, max_batch=2, max_tokens_per_seq=4400, kv_dtype=torch.bfloat16,
                rope_theta=5e5)
    base.update(kw)
    return pkv.StoreConfig(**base)


def prefill(store, cfg, host, seq, T):
    K, V = synth.prefill_kv(spec_of(cfg), T, seq=seq)  # unrotated keys
    store.load_prefill(seq, K.cuda(), V.cuda())
    host.set_prefill(seq, K, V)


def worst_err(store, cfg, host, seqs, layer, q, out):
    G = cfg.num_q_heads // cfg.num_kv_heads
    got = out.cpu().double().numpy()
    worst = 0.0
    for i, s in enumerate(seqs):
        for h in range(cfg.num_kv_heads):
            ref = oracle_decode_on_store(store, cfg, host, s, layer, h, q[i, h * G:(h + 1) * G].double().numpy())
            worst = max(worst, rel_err_rows(got[i, h * G:(h + 1) * G], ref))
    return worst


@pytest.mark.parametrize("P,d,rk,rv,theta,Hq", [(64, 128, 16, 24, 5e5, 8), (64, 128, 20, 12, 5e5, 8),
                                                 (32, 128, 16, 14, 5e5, 8), (64, 64, 24, 24, 1e4, 4),
                                                 (32, 64, 8, 8, 1e4, 8)])
def test_rope_store_decode_parity(pkv, P, d, rk, rv, theta, Hq):
    cfg = cfg_rope(pkv, page_size=P, head_dim=d, rank_k=rk, rank_v=rv, rope_theta=theta, num_q_heads=Hq,
                   recent_tokens=2 * P)
    store = pkv.Store(cfg)
    host = HostCache()
    prefill(store, cfg, host, 0, 4000)
    prefill(store, cfg, host, 1, 1500)
    q = synth.queries(2, cfg.num_q_heads, d, step=9, layer=1)
    out = torch.empty(2, cfg.num_q_heads, d, device="cuda")
    store.decode_attention(1, q.cuda(), out, [0, 1])
    assert store.check_device_status() == 0
    worst = worst_err(store, cfg, host, [0, 1], 1, q, out)
    print(f"rope P={P} d={d} ranks=({rk},{rv}) theta={theta:g} worst {worst:.3g}")
    assert worst <= TOL, worst


def test_rope_long_positions(pkv):
    """Angles up to 30000 rad on the fastest frequencies: the page-start table
    is computed in fp64 on the host."""
    cfg = cfg_rope(pkv, num_layers=1, max_batch=1, max_tokens_per_seq=30100)
    store = pkv.Store(cfg)
    host = HostCache()
    prefill(store, cfg, host, 0, 30000)
    q = synth.queries(1, cfg.num_q_heads, cfg.head_dim, step=2, layer=0)
    out = torch.empty(1, cfg.num_q_heads, cfg.head_dim, device="cuda")
    store.decode_attention(0, q.cuda(), out, [0])
    assert store.check_device_status() == 0
    worst = worst_err(store, cfg, host, [0], 0, q, out)
    print(f"rope T=30000 worst {worst:.3g}")
    assert worst <= TOL, worst


def test_rope_decode_steps_with_conversion(pkv):
    """decode_step across page boundaries: appended (unrotated) rows, the
    window page converted each 64 steps, every key turned at attention."""
    cfg = cfg_rope(pkv)
    store = pkv.Store(cfg)
    host = HostCache()
    spec = spec_of(cfg)
    prefill(store, cfg, host, 0, 1000)
    cache = {}
    worst = 0.0
    for step in range(160):
        for l in range(cfg.num_layers):
            T = len(torch.cat(host.k[(0, l, 0)]))
            k, v = synth.decode_tokens(spec, l, [0], [T], cache=cache)
            q = synth.queries(1, cfg.num_q_heads, cfg.head_dim, step=step, layer=l)
            out = torch.empty(1, cfg.num_q_heads, cfg.head_dim, device="cuda")
            store.decode_step(l, q.cuda(), k.cuda(), v.cuda(), out, [0])
            host.append(0, l, k[0], v[0])
            if step in (0, 40, 100, 159) and l == 1:
                worst = max(worst, worst_err(store, cfg, host, [0], l, q, out))
        store.convert_ready_pages()
    assert store.check_device_status() == 0
    for l in range(cfg.num_layers):
        check_page_table(store, cfg, 0, l, 1160)
    print(f"rope decode steps worst {worst:.3g}")
    assert worst <= TOL, worst
