"""The seeded input generators agree with themselves across their two entry
points (they hold none of the method's arithmetic)."""
import torch

import synth


def test_decode_rows_equal_decode_tokens():
    spec = synth.KVSpec(layers=2, kv_heads=2, head_dim=64, page_size=32, inner_rank=6, n_outliers=2,
                        rope_base=5e5)
    K, V = synth.decode_rows(spec, 1, 3, 100, 50)  # spans pages 3..4, RoPE at 100..149
    assert K.shape == (2, 50, 64) and V.shape == (2, 50, 64)
    cache = {}
    for j, pos in enumerate(range(100, 150)):
        k, v = synth.decode_tokens(spec, 1, [3], [pos], cache=cache)
        assert torch.equal(k[0], K[:, j]) and torch.equal(v[0], V[:, j]), pos
