"""decode_attn_host: the call with q, seq_lens and the block table in host
memory and out / lse returned to host memory (copies inside the call).  Its
results are bit-identical to decode_attn() at the same split count and match
the fp64 oracle; device status bits come back through the host word."""
import numpy as np
import pytest

import oracle
from split_kv_decode_attention_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_out_close, bf16_tensor_to_bits, to_device

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


def host_tensors(inp):
    """Pinned host copies of the per-call inputs (q bf16, block table, seq_lens)."""
    q = torch.from_numpy(np.ascontiguousarray(inp.q).view(np.int16)).view(torch.bfloat16)
    bt = None if inp.block_table is None else torch.from_numpy(
        np.ascontiguousarray(inp.block_table)).pin_memory()
    lens = torch.from_numpy(np.ascontiguousarray(inp.seq_lens)).pin_memory()
    return q.pin_memory(), bt, lens


CASES = [
    # name, batch, q_len, Hq, Hkv, lo, hi, paged, causal, fp8
    ("narrow_paged", 3, 1, 16, 4, 1, 900, True, False, False),
    ("narrow_contig_q4", 2, 4, 16, 4, 4, 700, False, True, False),
    ("wide64_paged", 3, 8, 64, 8, 8, 800, True, True, False),
    ("fp8_narrow", 3, 2, 16, 4, 2, 600, True, True, True),
    ("fp8_wide32", 2, 4, 32, 4, 4, 700, True, True, True),
]


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_entry_matches_device_entry_and_oracle(binding, case, splits):
    name, B, T, Hq, Hkv, lo, hi, paged, causal, fp8 = case
    shp = W.small_shape(name, batch=B, q_len=T, num_q_heads=Hq, num_kv_heads=Hkv, lo=lo, hi=hi,
                        paged=paged, causal=causal, seed=60 + B + T, kv_fp8=fp8)
    inp = W.make_host_inputs(shp)
    inp.seq_lens[0] = 0 if not causal else inp.seq_lens[0]   # an empty request where allowed
    q_d, k_d, v_d, bt_d, lens_d = to_device(inp)
    q_h, bt_h, lens_h = host_tensors(inp)
    p = binding.params_from_tensors(q_h, k_d, bt_h, max_seq_len=inp.max_seq_len, causal=causal,
                                    scale=shp.scale, k_scale=inp.k_scale, v_scale=inp.v_scale)
    S = splits if splits > 0 else binding.decode_attn_plan(p, inp.seq_lens)[0]
    out_h, lse_h, status = binding.decode_attn_host(
        q_h, k_d, v_d, bt_h, lens_h, max_seq_len=inp.max_seq_len, num_splits=splits, params=p)
    assert status == 0
    out_d, lse_d = binding.decode_attn(q_d, k_d, v_d, bt_d, lens_d, max_seq_len=inp.max_seq_len,
                                       num_splits=S, params=p)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_to_bits(out_h), bf16_tensor_to_bits(out_d))
    assert np.array_equal(lse_h.numpy().view(np.uint32), lse_d.cpu().numpy().view(np.uint32))
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(out_h.float().numpy().astype(np.float64), ref_o)
    assert_lse_close(lse_h.numpy(), ref_l)


def test_host_entry_reports_device_status(binding):
    """An out-of-range block-table entry: the DA_STATUS_BAD_PAGE bit comes
    back through the host status word of the same call."""
    shp = W.small_shape("host_status", batch=2, num_q_heads=8, num_kv_heads=2, lo=40, hi=90,
                        paged=True, seed=71)
    inp = W.make_host_inputs(shp)
    inp.block_table[1, 0] = inp.block_table.max() + 1000
    q_d, k_d, v_d, _, _ = to_device(inp)
    q_h, bt_h, lens_h = host_tensors(inp)
    _, _, status = binding.decode_attn_host(q_h, k_d, v_d, bt_h, lens_h,
                                            max_seq_len=inp.max_seq_len, num_splits=1)
    assert status & binding.DA_STATUS_BAD_PAGE
    # the next call with a good table reports nothing (the word is cleared per call)
    inp2 = W.make_host_inputs(shp)
    q_h, bt_h, lens_h = host_tensors(inp2)
    _, _, status = binding.decode_attn_host(q_h, k_d, v_d, bt_h, lens_h,
                                            max_seq_len=inp2.max_seq_len, num_splits=1)
    assert status == 0


@pytest.mark.parametrize("case", [CASES[0], CASES[2]], ids=[CASES[0][0], CASES[2][0]])
def test_host_entry_with_pageable_buffers(binding, case):
    """Ordinary (pageable) host tensors: the copies go through the driver's
    staging, and the results are bit-identical to the page-locked call."""
    name, B, T, Hq, Hkv, lo, hi, paged, causal, fp8 = case
    shp = W.small_shape(name, batch=B, q_len=T, num_q_heads=Hq, num_kv_heads=Hkv, lo=lo, hi=hi,
                        paged=paged, causal=causal, seed=80 + B + T, kv_fp8=fp8)
    inp = W.make_host_inputs(shp)
    _, k_d, v_d, _, _ = to_device(inp)
    q_h, bt_h, lens_h = host_tensors(inp)
    q_p = torch.from_numpy(np.ascontiguousarray(inp.q).view(np.int16)).view(torch.bfloat16)
    bt_p = None if inp.block_table is None else torch.from_numpy(
        np.ascontiguousarray(inp.block_table))
    lens_p = torch.from_numpy(np.ascontiguousarray(inp.seq_lens))
    out_p = torch.empty((B, T, Hq, 128), dtype=torch.bfloat16)
    lse_p = torch.empty((B, T, Hq), dtype=torch.float32)
    assert not q_p.is_pinned() and not out_p.is_pinned() and not lse_p.is_pinned()
    p = binding.params_from_tensors(q_h, k_d, bt_h, max_seq_len=inp.max_seq_len, causal=causal,
                                    scale=shp.scale)
    out_h, lse_h, st_h = binding.decode_attn_host(q_h, k_d, v_d, bt_h, lens_h,
                                                  max_seq_len=inp.max_seq_len, num_splits=3,
                                                  params=p)
    out_p, lse_p, st_p = binding.decode_attn_host(q_p, k_d, v_d, bt_p, lens_p,
                                                  max_seq_len=inp.max_seq_len, num_splits=3,
                                                  out_host=out_p, lse_host=lse_p, params=p)
    assert st_h == 0 and st_p == 0
    assert np.array_equal(bf16_tensor_to_bits(out_p), bf16_tensor_to_bits(out_h))
    assert np.array_equal(lse_p.numpy().view(np.uint32), lse_h.numpy().view(np.uint32))
