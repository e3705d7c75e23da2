"""INT4 factor stores [PuzzleKV §4.3] on the GPU.

Decode parity: the oracle decodes on the factors the store holds -- its 4-bit
codes times their fp16 scales, dequantized exactly in fp64 -- and the GPU's
outputs must agree within the bf16 bar, 2e-3 per row (decode on identical
factors).  The records themselves: codes in [-7, 7], every group's largest
element on +-7 (scale = max / 7), both factors carrying sigma^{1/2} (equal
column / row norms), and a reconstruction error as close to the page's own
optimum as the oracle's INT4 of its fp64 SVD gets.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import HostCache, check_page_table, oracle_decode_on_store, rel_err_rows, spec_of
from store_layout import Layout, factor_pool_slice, read_record, read_record_q4

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


def cfg_q4(pkv, **kw):
    base = dict(num_layers=2, num_kv_heads=2, num_q_heads=8, head_dim=128, page_size=64, rank_k=16, rank_v=24,
                sink_tokens=4, recent_tokens=128, max_batch=2, max_tokens_per_seq=4400, kv_dtype=torch.bfloat16,
                factor_int4=True)
    base.update(kw)
    return pkv.StoreConfig(**base)


def prefill(store, cfg, host, seq, T, rope=5e5):
    spec = spec_of(cfg, rope_base=rope)
    K, V = synth.prefill_kv(spec, T, seq=seq)
    store.load_prefill(seq, K.cuda(), V.cuda())
    host.set_prefill(seq, K, V)
    return spec


def check_decode(store, cfg, host, seqs, layer, q, out):
    G = cfg.num_q_heads // cfg.num_kv_heads
    got = out.cpu().double().numpy()
    worst = 0.0
    for i, s in enumerate(seqs):
        for h in range(cfg.num_kv_heads):
            ref = oracle_decode_on_store(store, cfg, host, s, layer, h, q[i, h * G:(h + 1) * G].double().numpy())
            worst = max(worst, rel_err_rows(got[i, h * G:(h + 1) * G], ref))
    assert worst <= TOL, worst
    return worst


@pytest.mark.parametrize("P,d,rk,rv", [(64, 128, 16, 24), (32, 128, 16, 14), (64, 64, 24, 24), (16, 64, 8, 8)])
def test_int4_store_decode_parity(pkv, P, d, rk, rv):
    cfg = cfg_q4(pkv, page_size=P, head_dim=d, rank_k=rk, rank_v=rv, recent_tokens=2 * P)
    store = pkv.Store(cfg)
    host = HostCache()
    prefill(store, cfg, host, 0, 4000)
    prefill(store, cfg, host, 1, 1500)
    for l in range(cfg.num_layers):
        check_page_table(store, cfg, 0, l, 4000)
    q = synth.queries(2, cfg.num_q_heads, d, step=9, layer=1)
    out = torch.empty(2, cfg.num_q_heads, d, device="cuda")
    store.decode_attention(1, q.cuda(), out, [0, 1])
    assert store.check_device_status() == 0
    print(f"int4 P={P} d={d} ranks=({rk},{rv}) worst {check_decode(store, cfg, host, [0, 1], 1, q, out):.3g}")


def test_int4_decode_steps_with_conversion(pkv):
    """decode_step across page boundaries with batched conversion on the
    store's internal stream: the converted pages' INT4 records are used."""
    cfg = cfg_q4(pkv)
    store = pkv.Store(cfg)
    host = HostCache()
    spec = prefill(store, cfg, host, 0, 1000)
    cache = {}
    for step in range(160):
        for l in range(cfg.num_layers):
            T = len(torch.cat(host.k[(0, l, 0)]))
            k, v = synth.decode_tokens(spec, l, [0], [T], cache=cache)
            q = synth.queries(1, cfg.num_q_heads, cfg.head_dim, step=step, layer=l)
            out = torch.empty(1, cfg.num_q_heads, cfg.head_dim, device="cuda")
            store.decode_step(l, q.cuda(), k.cuda(), v.cuda(), out, [0])
            host.append(0, l, k[0], v[0])
            if step in (0, 100, 159) and l == 1:
                check_decode(store, cfg, host, [0], l, q, out)
        store.convert_ready_pages()
    assert store.check_device_status() == 0
    for l in range(cfg.num_layers):
        check_page_table(store, cfg, 0, l, 1160)


def test_int4_records_quantize_absorbed_factors(pkv):
    cfg = cfg_q4(pkv, num_layers=1)
    store = pkv.Store(cfg)
    host = HostCache()
    prefill(store, cfg, host, 0, 3000)
    lay = Layout(cfg)
    kinds = oracle.page_kinds(3000, cfg.page_size, cfg.sink_tokens, cfg.recent_tokens)
    for h in range(cfg.num_kv_heads):
        fpool = factor_pool_slice(store, lay, 0, 0, h)
        Kh, Vh = host.rows(0, 0, h)
        for p in np.nonzero(kinds == oracle.FACTORED)[0][::7]:
            o = lay.record_offset(0, 0, h, int(p))
            rec = fpool[o:o + lay.rec_bytes]
            q = read_record_q4(rec, lay)
            assert np.all(q.pop("pad") == 0)  # the streams' unused registers hold code 0
            for name, (codes, scales, per_row) in q.items():
                assert codes.min() >= -7 and codes.max() <= 7
                groups = codes if per_row else codes.T
                for g, s in zip(groups, scales):
                    if s > 0:  # the group's largest element sits on +-7 (scale = max / 7 rounded to fp16)
                        assert np.abs(g).max() == 7, name
                    else:
                        assert np.all(g == 0), name
            LK, RK, LV, RV = read_record(rec, lay)
            for X, L, R, r, per_row_L in ((Kh, LK, RK, cfg.rank_k, False), (Vh, LV, RV, cfg.rank_v, True)):
                Xp = X[p * cfg.page_size:(p + 1) * cfg.page_size]
                # sigma^{1/2} on both sides: matching column / row norms, checked on the
                # components carrying most of the energy (the per-row scales of L_V are set
                # by a token's largest component, so small components quantize coarsely)
                cn, rn = np.linalg.norm(L, axis=0), np.linalg.norm(R, axis=1)
                big = rn >= 0.3 * rn.max()
                assert big.sum() >= 4 and np.all(np.abs(cn - rn)[big] <= 0.1 * rn[big])
                # reconstruction as good as the oracle's INT4 of the fp64 SVD
                err = np.linalg.norm(Xp - L @ R) / np.linalg.norm(Xp)
                Lo, Ro, _ = oracle.factorize(Xp, r)
                Lt, Rt = oracle.absorb_sigma(Lo, Ro)
                cL, sL = oracle.quantize_int4(Lt, per_row_L)
                cR, sR = oracle.quantize_int4(Rt, False)
                ref = oracle.dequantize_int4(cL, sL, per_row_L) @ oracle.dequantize_int4(cR, sR, False)
                err_o = np.linalg.norm(Xp - ref) / np.linalg.norm(Xp)
                assert err <= 1.15 * err_o + 1e-3 and err_o <= 1.15 * err + 1e-3, (err, err_o)


def expected_codes(x, per_row):
    """Codes and fp16 scales of the rule the records follow [PuzzleKV §4.3,
    readings C17-C18], in the kernel's fp32: scale = fp16(max|x| / 7) per
    group, code = round-half-to-even(x / scale) clamped to [-7, 7] (0 where
    the scale is 0)."""
    x = np.asarray(x, dtype=np.float32)
    m = np.abs(x).max(axis=1 if per_row else 0)
    s = (m / np.float32(7)).astype(np.float32).astype(np.float16).astype(np.float32)
    sb = s[:, None] if per_row else s[None, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.where(sb > 0, np.rint(x / np.where(sb > 0, sb, np.float32(1))), 0)
    return np.clip(c, -7, 7).astype(np.int64), s.astype(np.float64)


def kind_bytes(lay, kind):
    """Byte ranges of a record written by one kind's factorization job."""
    if kind == 0:
        return [(0, lay.q_off_V), (lay.q_off_sRK, lay.q_off_sRK + 2 * lay.d), (lay.q_off_sLK, lay.rec_bytes)]
    return [(lay.q_off_V, lay.q_off_sRK), (lay.q_off_sRV, lay.q_off_sRV + 2 * lay.d),
            (lay.q_off_sLV, lay.q_off_sLV + 2 * lay.P)]


@pytest.mark.parametrize("P,d,rk,rv", [(64, 128, 16, 24), (32, 128, 16, 14), (16, 64, 8, 8)])
def test_int4_codes_are_the_nearest_levels(pkv, P, d, rk, rv):
    """Integer work, checked exactly: every stored code is the nearest level
    x / s (ties to even, clamped to +-7) of the kernel's own absorbed fp32
    factor x and the record's own fp16 scale s, and every scale is
    fp16(max |x| / 7) of its group (columns of L~_K, R~_K and R~_V, rows of
    L~_V).  The store's records of the same pages are byte for byte the
    stateless call's."""
    cfg = cfg_q4(pkv, page_size=P, head_dim=d, rank_k=rk, rank_v=rv, num_layers=1, recent_tokens=2 * P)
    lay = Layout(cfg)
    assert pkv.int4_record_bytes(P, d, rk, rv) == lay.rec_bytes
    T = 30 * P
    store = pkv.Store(cfg)
    host = HostCache()
    prefill(store, cfg, host, 0, T)
    kinds = oracle.page_kinds(T, P, cfg.sink_tokens, cfg.recent_tokens)
    fac = [int(p) for p in np.nonzero(kinds == oracle.FACTORED)[0]]
    for kind, r in ((0, rk), (1, rv)):
        X = torch.tensor(np.stack([host.rows(0, 0, h)[kind][p * P:(p + 1) * P] for h in range(cfg.num_kv_heads)
                                   for p in fac]), dtype=torch.bfloat16, device="cuda")
        rec, Lq, Rq, st = pkv.factorize_batch_int4(X, rk, rv, kind)
        assert int(st.item()) == 0
        rec, Lq, Rq = rec.cpu().numpy(), Lq.cpu().numpy(), Rq.cpu().numpy()
        i = 0
        for h in range(cfg.num_kv_heads):
            fpool = factor_pool_slice(store, lay, 0, 0, h)
            for p in fac:
                q = read_record_q4(rec[i], lay)
                if kind == 0:
                    parts = ((q["LK"], Lq[i], False), (q["RK"], Rq[i], False))
                else:  # stored transposed: L_V as [rank][token] (groups = tokens), R_V as [dim][rank]
                    parts = ((q["LVt"], Lq[i].T, False), (q["RVt"], Rq[i].T, True))
                for (codes, scales, per_row), x, per_row_x in parts:
                    assert per_row == per_row_x
                    want_c, want_s = expected_codes(x, per_row)
                    assert np.array_equal(scales, want_s), (kind, h, p)
                    assert np.array_equal(codes.astype(np.int64), want_c), (kind, h, p)
                o = lay.record_offset(0, 0, h, p)
                for a, b in kind_bytes(lay, kind):
                    assert np.array_equal(fpool[o + a:o + b], rec[i][a:b]), (kind, h, p, a)
                i += 1
