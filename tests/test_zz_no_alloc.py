"""The allocation-free decode entry point (split-K scratch in the library's
static device array) against the regular entry point (scratch in the store's
workspace).  Collected last so that a failure here, in a run that stops at
the first failure, comes after every other test has run.

Callers that need it cannot allocate device memory where they decode, e.g.
runtimes that forbid allocation once serving has started."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from page_wise_rank_gb300 import build
    build.build()
    import page_wise_rank_gb300 as m
    return m


def rel_err_rows(a, b):
    a, b = a.reshape(-1, a.shape[-1]), b.reshape(-1, b.shape[-1])
    return float((np.abs(a - b).max(axis=1) / np.abs(b).max(axis=1)).max())


def test_static_scratch_decode_matches_workspace_decode(pkv):
    cfg = pkv.StoreConfig(num_layers=2, num_kv_heads=4, num_q_heads=16, head_dim=128, page_size=64, rank_k=16,
                          rank_v=24, sink_tokens=4, recent_tokens=128, max_batch=3, max_tokens_per_seq=5000,
                          kv_dtype=torch.bfloat16)
    spec = synth.KVSpec(layers=2, kv_heads=4, head_dim=128, page_size=64, inner_rank=12, n_outliers=4,
                        rope_base=5e5, dtype=torch.bfloat16)
    store = pkv.Store(cfg)
    for seq, T in ((0, 4321), (2, 900)):
        K, V = synth.prefill_kv(spec, T, seq=seq)
        store.load_prefill(seq, K.cuda(), V.cuda())
    q = synth.queries(2, 16, 128, step=9, layer=1).cuda()
    ref = torch.empty(2, 16, 128, device="cuda")
    store.decode_attention(1, q, ref, [2, 0])
    assert store.check_device_status() == 0
    outs = [torch.full((2, 16, 128), float("nan"), device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free = []
    for out in outs:  # two calls in a row: the array keeps the last call's contents
        free.append(torch.cuda.mem_get_info()[0])
        store.decode_attention_static_scratch(1, q, out, [2, 0])
        assert store.check_device_status() == 0
        # the same kernel on the same inputs, merging the splits in the same
        # order: bitwise equal to the workspace path
        assert rel_err_rows(out.cpu().double().numpy(), ref.cpu().double().numpy()) <= 2e-3
        assert torch.equal(out, ref)
    # the first call may load the library's device code and its array; after
    # that the call takes no device memory
    assert torch.cuda.mem_get_info()[0] == free[1]


def test_static_scratch_rejects_oversized_store(pkv):
    cfg = pkv.StoreConfig(num_layers=1, num_kv_heads=8, num_q_heads=64, head_dim=128, page_size=64, rank_k=16,
                          rank_v=16, sink_tokens=4, recent_tokens=128, max_batch=8, max_tokens_per_seq=256,
                          kv_dtype=torch.bfloat16)
    store = pkv.Store(cfg)
    spec = synth.KVSpec(layers=1, kv_heads=8, head_dim=128, page_size=64, dtype=torch.bfloat16)
    K, V = synth.prefill_kv(spec, 200)
    store.load_prefill(0, K.cuda(), V.cuda())
    q = torch.zeros(1, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(1, 64, 128, device="cuda")
    with pytest.raises(pkv.PuzzleKVError) as e:
        store.decode_attention_static_scratch(0, q, out, [0])
    assert e.value.status == 3 and "16777216" in str(e.value)
