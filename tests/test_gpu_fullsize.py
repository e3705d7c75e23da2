"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: one decode_step launch per layer, issued back to back on
one stream, with the batched page conversion between decode steps.

The oracle decodes sampled (sequence, layer, KV head) triples in fp64 on the
factors the GPU stored (copied back and upcast exactly) and on the dense rows
the store was fed; per output row the max relative error must stay within
2e-3 (bf16 storage, decode on identical factors).  Page tables are checked
bit-exactly against the oracle's classification.  Inputs are the seeded
synthetic caches, generated on the GPU; only the sampled slices come back to
the host.

Workloads:
  * Llama-3.1-8B-shaped attention, 32 layers, 8 KV / 32 query heads, d = 128,
    T = 32768, P = 64, r_K = 16, r_V = 24, sink 4, recent 128, RoPE keys.
  * Batched serving decode, same shapes, 16 requests of U[8K, 32K] tokens
    (seed 7), ragged page tables; 4 layers (every layer's launch is the same).
  * Qwen3-32B-shaped attention, 64 layers, 8 KV / 64 query heads,
    T = 131072, r_K = r_V = 24: whole-cache factorization, then 32 steps.
  * Incremental compression during generation: Llama shapes, batch 8,
    4096-token prompts, 4096 decode steps with pages converted on the decode
    stream as they complete.
  * The Llama shape at T = 32768 with INT4 factor records (PuzzleKV §4.3;
    the oracle decodes the exactly dequantized codes), with the pages' own
    P = 32, (r_K, r_V) = (16, 14) and a 64-token window, and with keys stored
    before RoPE (theta 5e5) and turned at attention (PuzzleKV §4.1).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import rel_err_rows, spec_of
from store_layout import Layout, descriptors, lengths, read_record

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


def llama_cfg(pkv, layers, B, Tmax, **kw):
    base = dict(num_layers=layers, num_kv_heads=8, num_q_heads=32, head_dim=128, page_size=64, rank_k=16,
                rank_v=24, sink_tokens=4, recent_tokens=128, max_batch=B, max_tokens_per_seq=Tmax,
                kv_dtype=torch.bfloat16)
    base.update(kw)
    return pkv.StoreConfig(**base)


def oracle_err(store, cfg, K, V, q_rows, got_rows, seq, layer, h):
    """Max row error of the GPU output of KV head h against the oracle run on
    the store's factors (K, V: [T, d] rows fed to the store, fp64)."""
    T, P = K.shape[0], cfg.page_size
    kinds = oracle.page_kinds(T, P, cfg.sink_tokens, cfg.recent_tokens)
    n = len(kinds)
    lay = Layout(cfg)
    o0 = lay.record_offset(layer, seq, h, 0)
    raw = store.factor_pool[o0:o0 + n * lay.rec_bytes].cpu().numpy()
    LK, RK = np.zeros((n, P, cfg.rank_k)), np.zeros((n, cfg.rank_k, cfg.head_dim))
    LV, RV = np.zeros((n, P, cfg.rank_v)), np.zeros((n, cfg.rank_v, cfg.head_dim))
    for p in np.nonzero(kinds == oracle.FACTORED)[0]:
        LK[p], RK[p], LV[p], RV[p] = read_record(raw[p * lay.rec_bytes:(p + 1) * lay.rec_bytes], lay)
    theta = float(getattr(cfg, "rope_theta", 0.0))
    if theta > 0:  # keys stored before RoPE: the oracle turns them at their positions too
        ref = oracle.decode_head_rope(q_rows, kinds, K, V, LK, RK, LV, RV, T, P, theta)
    else:
        ref = oracle.decode_head(q_rows, kinds, K, V, LK, RK, LV, RV, T, P)
    return rel_err_rows(got_rows, ref)


def check_table(store, cfg, seq, layer, T):
    lay = Layout(cfg)
    assert lengths(store, lay)[seq, layer] == T
    n = (T + cfg.page_size - 1) // cfg.page_size
    kinds, slots = descriptors(store, lay, seq, layer, n)
    assert np.array_equal(kinds, oracle.page_kinds(T, cfg.page_size, cfg.sink_tokens, cfg.recent_tokens))
    fac = kinds == oracle.FACTORED
    assert np.array_equal(slots[fac], np.nonzero(fac)[0])


def run_steps(store, cfg, spec, seqs, T0, steps, samples, prefill_rows, q_of, check_steps):
    """decode_step over every layer for `steps` steps, back to back per step
    (inputs staged on the device first), batched conversion after each step;
    returns the worst sampled error over check_steps."""
    L, B = cfg.num_layers, len(seqs)
    G = cfg.num_q_heads // cfg.num_kv_heads
    # decode-phase rows of every (layer, seq): [L, steps, B, H, d] on the device
    kdec = torch.empty(L, steps, B, cfg.num_kv_heads, cfg.head_dim, dtype=cfg.kv_dtype, device="cuda")
    vdec = torch.empty_like(kdec)
    for l in range(L):
        for i, s in enumerate(seqs):
            k, v = synth.decode_rows(spec, l, s, T0[i], steps, device="cuda")
            kdec[l, :, i] = k.transpose(0, 1)
            vdec[l, :, i] = v.transpose(0, 1)
    out = torch.empty(L, B, cfg.num_q_heads, cfg.head_dim, dtype=torch.float32, device="cuda")
    worst = 0.0
    for step in range(steps):
        for l in range(L):
            store.decode_step(l, q_of(step, l), kdec[l, step], vdec[l, step], out[l], seqs)
        store.convert_ready_pages()
        if step in check_steps:
            assert store.check_device_status() == 0
            got = out.cpu().double().numpy()
            for (i, l, h) in samples:
                s = seqs[i]
                K = np.concatenate([prefill_rows[(i, l, h)][0],
                                    kdec[l, :step + 1, i, h].cpu().double().numpy()])
                V = np.concatenate([prefill_rows[(i, l, h)][1],
                                    vdec[l, :step + 1, i, h].cpu().double().numpy()])
                q = q_of(step, l)[i, h * G:(h + 1) * G].cpu().double().numpy()
                err = oracle_err(store, cfg, K, V, q, got[l, i, h * G:(h + 1) * G], s, l, h)
                assert err <= TOL, (step, i, l, h, err)
                worst = max(worst, err)
    assert store.check_device_status() == 0
    return worst


def prefill_seq(store, spec, seq, T, samples_for_seq, rows, index):
    K, V = synth.prefill_kv(spec, T, seq=seq, device="cuda")
    store.load_prefill(seq, K, V)
    for (l, h) in samples_for_seq:
        rows[(index, l, h)] = (K[l, h].double().cpu().numpy(), V[l, h].double().cpu().numpy())
    del K, V


def make_q(cfg, B, n_distinct=8):
    """Per (step, layer) queries: n_distinct seeded sets per layer, reused cyclically."""
    qs = [[synth.queries(B, cfg.num_q_heads, cfg.head_dim, step=s, layer=l, dtype=cfg.kv_dtype).cuda()
           for l in range(cfg.num_layers)] for s in range(n_distinct)]
    return lambda step, l: qs[step % n_distinct][l]


def test_llama32k_full_size(pkv):
    T0 = 32768
    cfg = llama_cfg(pkv, 32, 1, T0 + 64)
    spec = spec_of(cfg, inner_rank=12, n_outliers=4, rope_base=5e5)
    store = pkv.Store(cfg)
    samples = [(0, 0, 0), (0, 17, 5), (0, 31, 7)]
    rows = {}
    prefill_seq(store, spec, 0, T0, [(l, h) for _, l, h in samples], rows, 0)
    worst = run_steps(store, cfg, spec, [0], [T0], 3, samples, rows, make_q(cfg, 1), check_steps={0, 2})
    for l in (0, 31):
        check_table(store, cfg, 0, l, T0 + 3)
    print("llama32k worst", worst)


def test_batched16_ragged_full_size(pkv):
    lens = synth.batch_lengths(16, 8192, 32768, seed=7)
    cfg = llama_cfg(pkv, 4, 16, max(lens) + 64)
    spec = spec_of(cfg, inner_rank=12, n_outliers=4, rope_base=5e5)
    store = pkv.Store(cfg)
    sample_seqs = (0, 5, 11, 15)
    samples = [(i, l, h) for i in sample_seqs for l in (0, 3) for h in (0, 7)]
    rows = {}
    for i, T in enumerate(lens):
        prefill_seq(store, spec, i, T, [(l, h) for j, l, h in samples if j == i], rows, i)
    seqs = list(range(16))
    worst = run_steps(store, cfg, spec, seqs, lens, 2, samples, rows, make_q(cfg, 16), check_steps={1})
    for i in sample_seqs:
        check_table(store, cfg, i, 3, lens[i] + 2)
    print("batched16 worst", worst)


def test_qwen128k_full_size(pkv):
    T0 = 131072
    cfg = pkv.StoreConfig(num_layers=64, num_kv_heads=8, num_q_heads=64, head_dim=128, page_size=64, rank_k=24,
                          rank_v=24, sink_tokens=4, recent_tokens=128, max_batch=1, max_tokens_per_seq=T0 + 64,
                          kv_dtype=torch.bfloat16)
    spec = spec_of(cfg, inner_rank=12, n_outliers=4)
    store = pkv.Store(cfg)
    samples = [(0, 0, 0), (0, 40, 3), (0, 63, 7)]
    rows = {}
    prefill_seq(store, spec, 0, T0, [(l, h) for _, l, h in samples], rows, 0)
    worst = run_steps(store, cfg, spec, [0], [T0], 32, samples, rows, make_q(cfg, 1), check_steps={31})
    check_table(store, cfg, 0, 63, T0 + 32)
    print("qwen128k worst", worst)


def test_incremental_4096_steps_batch8(pkv):
    T0, steps, B = 4096, 4096, 8
    cfg = llama_cfg(pkv, 32, B, T0 + steps + 64)
    spec = spec_of(cfg, inner_rank=12, n_outliers=4, rope_base=5e5)
    store = pkv.Store(cfg)
    samples = [(0, 0, 0), (3, 9, 4), (7, 31, 7)]
    rows = {}
    for i in range(B):
        prefill_seq(store, spec, i, T0, [(l, h) for j, l, h in samples if j == i], rows, i)
    worst = run_steps(store, cfg, spec, list(range(B)), [T0] * B, steps, samples, rows, make_q(cfg, B),
                      check_steps={0, 2047, steps - 1})
    for i, l, _ in samples:
        check_table(store, cfg, i, l, T0 + steps)
    print("incremental worst", worst)


@pytest.mark.parametrize("variant", ["int4", "p32", "prerope"])
def test_llama32k_variants_full_size(pkv, variant):
    T0 = 32768
    rope = 5e5
    if variant == "int4":
        kw = dict(factor_int4=True)
    elif variant == "p32":
        kw = dict(page_size=32, rank_k=16, rank_v=14, recent_tokens=64)
    else:  # keys given before RoPE: the store turns them, the generator leaves them unrotated
        kw = dict(rope_theta=5e5)
        rope = None
    cfg = llama_cfg(pkv, 32, 1, T0 + 64, **kw)
    spec = spec_of(cfg, inner_rank=12, n_outliers=4, rope_base=rope)
    store = pkv.Store(cfg)
    samples = [(0, 0, 0), (0, 31, 7)]
    rows = {}
    prefill_seq(store, spec, 0, T0, [(l, h) for _, l, h in samples], rows, 0)
    worst = run_steps(store, cfg, spec, [0], [T0], 2, samples, rows, make_q(cfg, 1), check_steps={1})
    check_table(store, cfg, 0, 31, T0 + 2)
    print(variant, "worst", worst)
