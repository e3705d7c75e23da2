"""Layer-by-layer prefill compression [PuzzleKV §3.3 ①②③, §4.5 time to first token].

puzzlekv_factorize_layer runs the same kernels as the whole-prompt
puzzlekv_load_prefill, restricted to one layer; in the background form the
factorization runs on the store's internal stream while the caller's stream
goes on.  Both must leave the store byte for byte as the whole-prompt call
does (the factorization and the page-table writes are deterministic), and
decode on either store must give bitwise equal outputs -- whether or not the
caller waits for the background work first, since decode waits for it.
Stores filled layer by layer are also checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import HostCache, oracle_decode_on_store, rel_err_rows, spec_of
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
    ref.load_prefill(1, K, V)
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
    ref.load_prefill(0, K, V)
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


@pytest.mark.parametrize("int4", [False, True])
@pytest.mark.parametrize("background", [False, True])
def test_layer_prefill_against_oracle(pkv, int4, background):
    """Stores filled layer by layer, inline and in the background, checked
    against the oracle: decode on the stored factors equals the oracle's
    attention on the same factors (C6, 2e-3 per output row), with no explicit
    wait for the background work.  bf16 records are the kernel's own factors
    of the prompt pages: equal to the stateless factorization of the same
    pages rounded to bf16, whose fp32 form is within 1e-3 of the oracle's
    rank-r optimum on every page (C5)."""
    cfg = cfg_of(pkv, factor_int4=int4)
    T, P = 3000, cfg.page_size
    K, V = synth.prefill_kv(spec_of(cfg, rope_base=5e5), T, seq=0)
    host = HostCache()
    host.set_prefill(0, K, V)
    st = pkv.Store(cfg)
    Kd, Vd = K.cuda(), V.cuda()
    for l in range(cfg.num_layers):
        st.factorize_layer(0, l, Kd[l].clone(), Vd[l].clone(), background=background)
    G = cfg.num_q_heads // cfg.num_kv_heads
    for l in (0, cfg.num_layers - 1):
        q = synth.queries(1, cfg.num_q_heads, cfg.head_dim, step=5, layer=l)
        out = torch.empty(1, cfg.num_q_heads, cfg.head_dim, device="cuda")
        st.decode_attention(l, q.cuda(), out, [0])
        assert st.check_device_status() == 0, pkv.last_error()
        got = out.cpu().double().numpy()[0]
        for h in range(cfg.num_kv_heads):
            ref = oracle_decode_on_store(st, cfg, host, 0, l, h, q[0, h * G:(h + 1) * G].double().numpy())
            assert rel_err_rows(got[h * G:(h + 1) * G], ref) <= 2e-3, (l, h)
    if int4:
        return
    lay = Layout(cfg)
    l = 2
    kinds = oracle.page_kinds(T, P, cfg.sink_tokens, cfg.recent_tokens)
    fac = np.nonzero(kinds == oracle.FACTORED)[0]
    fpool = st.factor_pool.cpu().numpy()
    for kind, src, r in ((0, Kd, cfg.rank_k), (1, Vd, cfg.rank_v)):
        X = torch.stack([src[l, h, p * P:(p + 1) * P] for h in range(cfg.num_kv_heads) for p in fac])
        Lb, Rb, _, s1 = pkv.factorize_batch(X, r, out_dtype=torch.bfloat16, sigma=False)
        Lf, Rf, _, s2 = pkv.factorize_batch(X, r, out_dtype=torch.float32, sigma=False)
        assert int(s1.item()) == 0 and int(s2.item()) == 0
        Lb, Rb = Lb.double().cpu().numpy(), Rb.double().cpu().numpy()
        Lf, Rf = Lf.double().cpu().numpy(), Rf.double().cpu().numpy()
        Xh = X.double().cpu().numpy()
        i = 0
        for h in range(cfg.num_kv_heads):
            for p in fac:
                f = read_factors(fpool, lay, l, 0, h, int(p))
                Ls, Rs = (f[0], f[1]) if kind == 0 else (f[2], f[3])
                assert np.array_equal(Ls, Lb[i]) and np.array_equal(Rs, Rb[i]), (kind, h, p)
                _, _, S = oracle.factorize(Xh[i], r)
                e_opt = np.sqrt(np.sum(S[r:] ** 2))
                e = np.linalg.norm(Xh[i] - Lf[i] @ Rf[i])
                assert (e - e_opt) / e_opt <= 1e-3, (kind, h, p, e, e_opt)
                i += 1
