"""Seeded random shapes through the C ABI against the fp64 oracle: GQA group
and draft-token count on both kernels (1..128 rows per KV head; a second set
draws only 17..128 rows, the tcgen05 kernel's), paged caches
of 16 / 32 / 64-token pages and contiguous ones, bf16 and FP8 E4M3 caches,
causal or not, explicit and planned split counts, one-launch and two-pass
forms.  Each case is small enough for the oracle and spans several tiles,
stages and chunks with ragged tails."""
import numpy as np
import pytest

import oracle
from split_kv_decode_attention_gb300 import workloads as W
from tests.parity import (assert_lse_close, assert_out_close, assert_ulps_close,
                          bf16_tensor_to_bits, bf16_tensor_to_f64, to_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from split_kv_decode_attention_gb300 import binding as B
    from split_kv_decode_attention_gb300 import build as cuda_build
    cuda_build.build()
    B.lib()
    return B


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    while True:
        G = int(rng.choice([1, 2, 4, 8, 16]))
        q_len = int(rng.integers(1, 9))
        if G * q_len <= 128:
            break
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 6))
    causal = bool(q_len > 1 and rng.random() < 0.7)
    lo = q_len if causal else int(rng.integers(0, 40))
    hi = int(rng.integers(max(lo, 1) + 1, 1500))
    paged = bool(rng.random() < 0.7)
    page = int(rng.choice([16, 32, 64])) if paged else 16
    fp8 = bool(rng.random() < 0.35)
    splits = int(rng.choice([0, 1, int(rng.integers(2, 21))]))
    two_pass = bool(rng.random() < 0.3)
    shp = W.small_shape(f"rand{seed}", batch=B, q_len=q_len, num_q_heads=G * Hkv,
                        num_kv_heads=Hkv, lo=lo, hi=hi, paged=paged, page_size=page,
                        causal=causal, seed=2000 + seed, kv_fp8=fp8)
    return shp, splits, two_pass


@pytest.mark.parametrize("seed", range(96))
def test_random_shape_matches_oracle(binding, seed):
    shp, splits, two_pass = draw_case(seed)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len,
                                   causal=shp.causal, scale=shp.scale, num_splits=splits,
                                   status=status, two_pass=two_pass,
                                   k_scale=inp.k_scale, v_scale=inp.v_scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, (shp, splits, two_pass)
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o, what=f"out {shp.name}")
    assert_lse_close(lse.cpu().numpy(), ref_l, what=f"lse {shp.name}")
    assert_ulps_close(bf16_tensor_to_bits(out), ref_o, what=f"out {shp.name}")


def draw_wide_case(seed):
    """17..128 rows per KV head (the tcgen05 kernel, key-split below 65 rows),
    up to 8 requests of up to 3000 tokens."""
    rng = np.random.default_rng(7000 + seed)
    while True:
        G = int(rng.choice([4, 8, 16, 32]))
        q_len = int(rng.integers(1, 9))
        if 16 < G * q_len <= 128:
            break
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 9))
    causal = bool(q_len > 1 and rng.random() < 0.7)
    lo = q_len if causal else int(rng.integers(0, 40))
    hi = int(rng.integers(max(lo, 1) + 1, 3000))
    paged = bool(rng.random() < 0.7)
    page = int(rng.choice([16, 32, 64])) if paged else 16
    fp8 = bool(rng.random() < 0.4)
    splits = int(rng.choice([0, 1, int(rng.integers(2, 9))]))
    two_pass = bool(rng.random() < 0.3)
    shp = W.small_shape(f"wide{seed}", batch=B, q_len=q_len, num_q_heads=G * Hkv,
                        num_kv_heads=Hkv, lo=lo, hi=hi, paged=paged, page_size=page,
                        causal=causal, seed=8000 + seed, kv_fp8=fp8)
    return shp, splits, two_pass


@pytest.mark.parametrize("seed", range(48))
def test_random_wide_shape_matches_oracle(binding, seed):
    shp, splits, two_pass = draw_wide_case(seed)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len,
                                   causal=shp.causal, scale=shp.scale, num_splits=splits,
                                   status=status, two_pass=two_pass,
                                   k_scale=inp.k_scale, v_scale=inp.v_scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, (shp, splits, two_pass)
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o, what=f"out {shp.name}")
    assert_lse_close(lse.cpu().numpy(), ref_l, what=f"lse {shp.name}")
    assert_ulps_close(bf16_tensor_to_bits(out), ref_o, what=f"out {shp.name}")
