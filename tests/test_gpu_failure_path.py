"""Failure detection of the decode kernel, exercised without a GPU fault.

Every wait of the kernel is bounded; a wait that runs out sets the device
status word, lets the CTA's copies land and ends the CTA without its result,
and the host learns of it from puzzlekv_check_device_status, which also
clears the split tickets so that the store keeps working.  The test hook
makes one shared-memory barrier expect 16 bytes that no copy delivers (a
flag nothing sets) and shortens the waits of that one launch to 50 us.
"""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import HostCache, oracle_decode_on_store, rel_err_rows, spec_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from page_wise_rank_gb300 import build
    build.build()
    import page_wise_rank_gb300 as m
    return m


@pytest.fixture(scope="module")
def loaded(pkv):
    # 8 KV heads: few enough splits per head that the merge stages their
    # states in shared memory (the barrier the merge hook poisons)
    cfg = pkv.StoreConfig(num_layers=1, num_kv_heads=8, num_q_heads=32, head_dim=128, page_size=64, rank_k=16,
                          rank_v=24, sink_tokens=4, recent_tokens=128, max_batch=1, max_tokens_per_seq=8192,
                          kv_dtype=torch.bfloat16)
    store = pkv.Store(cfg)
    host = HostCache()
    K, V = synth.prefill_kv(spec_of(cfg, rope_base=5e5), 7000, seq=0)
    store.load_prefill(0, K.cuda(), V.cuda())
    host.set_prefill(0, K, V)
    q = synth.queries(1, 32, 128, step=0, dtype=torch.bfloat16)
    refs = [oracle_decode_on_store(store, cfg, host, 0, 0, h, q[0, 4 * h:4 * h + 4].double().numpy())
            for h in range(8)]
    return store, q.cuda(), refs


def decode(store, q):
    out = torch.full((1, 32, 128), float("nan"), device="cuda")
    store.decode_attention(0, q, out, [0])
    return out


def assert_matches(out, refs, heads=range(8)):
    got = out.cpu().double().numpy()[0]
    for h in heads:
        assert rel_err_rows(got[4 * h:4 * h + 4], refs[h]) <= 2e-3


def test_unit_wait_runs_out(pkv, loaded):
    """The first unit of the first CTA of KV head 0 never completes: that CTA
    gives up, KV head 0's output rows stay unwritten, the others' are right,
    the status reports the timeout, and the next decode is right again."""
    store, q, refs = loaded
    store.debug_fail_next_wait(1, 50_000)
    out = decode(store, q)
    assert store.check_device_status() == pkv._lib.ERR_DEVICE_TIMEOUT
    assert torch.isnan(out[0, :4]).all()
    assert_matches(out, refs, heads=range(1, 8))
    out = decode(store, q)
    assert store.check_device_status() == 0, pkv.last_error()
    assert_matches(out, refs)


def test_merge_wait_runs_out(pkv, loaded):
    """The split merge never gets its copies: no output row is written, the
    status reports the timeout, and the next decode is right again."""
    store, q, refs = loaded
    store.debug_fail_next_wait(2, 50_000)
    out = decode(store, q)
    assert store.check_device_status() == pkv._lib.ERR_DEVICE_TIMEOUT
    assert torch.isnan(out).all()
    for _ in range(2):
        out = decode(store, q)
        assert store.check_device_status() == 0, pkv.last_error()
        assert_matches(out, refs)


def test_hook_applies_to_one_launch(pkv, loaded):
    store, q, refs = loaded
    store.debug_fail_next_wait(2, 50_000)
    store.debug_fail_next_wait(0, 50_000)  # cleared before any launch
    out = decode(store, q)
    assert store.check_device_status() == 0
    assert_matches(out, refs)
    with pytest.raises(pkv.PuzzleKVError):
        store.debug_fail_next_wait(3, 50_000)
    with pytest.raises(pkv.PuzzleKVError):
        store.debug_fail_next_wait(1, 10)
