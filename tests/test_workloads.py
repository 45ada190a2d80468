"""The seeded input generator: bf16 rounding, length mix and block tables."""
import numpy as np
import torch

from split_kv_decode_attention_gb300 import workloads as W


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8,
                                  np.inf, -np.inf, 3.4e38], np.float32)])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_block_table_is_a_permutation_with_unused_slots_minus_one():
    shp = W.WORKLOADS["c3_b64_h32kv8_L512-32768_paged"]
    rng = np.random.default_rng(shp.seed)
    lens = W.draw_seq_lens(shp, rng)
    assert lens.min() >= 512 and lens.max() <= 32768
    bt, P = W.draw_block_table(lens, 16, 32768 // 16, rng)
    need = (lens + 15) // 16
    assert P == need.sum()
    used = np.concatenate([bt[b, :n] for b, n in enumerate(need)])
    np.testing.assert_array_equal(np.sort(used), np.arange(P))
    for b, n in enumerate(need):
        assert np.all(bt[b, n:] == -1)


def test_small_host_inputs_shapes_and_determinism():
    shp = W.small_shape(batch=4, q_len=2, num_q_heads=8, num_kv_heads=2,
                        lo=3, hi=70, causal=True, peaked=0.05)
    a = W.make_host_inputs(shp)
    b = W.make_host_inputs(shp)
    np.testing.assert_array_equal(a.k_cache, b.k_cache)
    np.testing.assert_array_equal(a.block_table, b.block_table)
    assert a.q.shape == (4, 2, 8, 128) and a.q.dtype == np.uint16
    assert a.k_cache.shape[1:] == (16, 2, 128)
    assert a.kv_bytes() == int(a.seq_lens.sum()) * 2 * 128 * 4
