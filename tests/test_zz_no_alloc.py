"""decode_attn_static_workspace(): decode attention for callers that cannot
allocate device memory (plugin hosts that pass only input/output buffers,
runtimes whose memory belongs to another allocator, deployments that forbid
allocation after start-up).  Its partials live in the library's fixed 16 MiB
device array instead of a caller workspace.

Checked through the C ABI against decode_attn() with a caller workspace, on
two calls in a row.  The calls are forced onto the two-launch path (split
kernel writing fp32 partials, then the combine kernel), so the partials really
go through the static array; the first call of each pair writes more splits
and rows than the second, so the second runs over larger stale data the first
left there.  Same kernels and same splits give identical bits, so the outputs
are compared bit for bit (and, redundantly, within the parity tolerance).
This file is collected last so that a stop-at-first-failure run has already
run the rest; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest

from split_kv_decode_attention_gb300 import workloads as W
from tests.parity import (assert_lse_close, assert_out_close, bf16_tensor_to_bits,
                          bf16_tensor_to_f64, to_device)

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


def both_ways(binding, inp, num_splits):
    """decode_attn_static_workspace and decode_attn (caller workspace) on the
    same inputs, both on the two-launch path; returns (static out bits,
    static lse, reference out bits, reference lse, reference out values)."""
    q, k, v, bt, lens = to_device(inp)
    s = inp.shape
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=s.causal,
                                    scale=s.scale, k_scale=inp.k_scale, v_scale=inp.v_scale,
                                    two_pass=True)
    assert binding.decode_attn_launch_count(p, num_splits) == 2
    assert binding.decode_attn_workspace_bytes(p, num_splits) > 0
    ref_out, ref_lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len,
                                           causal=s.causal, scale=s.scale,
                                           num_splits=num_splits, params=p)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.decode_attn_static_workspace(p, q, k, v, bt, lens, out, lse, num_splits,
                                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (bf16_tensor_to_bits(out), lse.cpu().numpy(), bf16_tensor_to_bits(ref_out),
            ref_lse.cpu().numpy(), bf16_tensor_to_f64(out), bf16_tensor_to_f64(ref_out))


def check_pair(binding, calls):
    for inp, splits in calls:
        out_b, lse, ref_b, ref_lse, out_f, ref_f = both_ways(binding, inp, splits)
        assert np.array_equal(out_b, ref_b), "static-workspace out differs from decode_attn"
        assert np.array_equal(lse.view(np.uint32), ref_lse.view(np.uint32)), \
            "static-workspace lse differs from decode_attn"
        assert_out_close(out_f, ref_f, what="static-workspace out")
        assert_lse_close(lse, ref_lse, what="static-workspace lse")


def test_two_calls_in_a_row_match_decode_attn(binding):
    """Warp-MMA kernel: 16 rows per KV head and 9 splits, then 8 rows and 3
    splits over the first call's leftovers."""
    first = W.make_host_inputs(W.small_shape(
        "na1", batch=5, q_len=4, num_q_heads=16, num_kv_heads=4, lo=300, hi=3000,
        paged=True, causal=True, seed=91))
    second = W.make_host_inputs(W.small_shape(
        "na2", batch=2, q_len=1, num_q_heads=8, num_kv_heads=1, lo=900, hi=1200,
        paged=False, seed=92))
    check_pair(binding, ((first, 9), (second, 3)))


def test_fp8_and_wide_calls_match_decode_attn(binding):
    """FP8 caches (warp-MMA kernel), then a 64-row query group on the tcgen05
    kernel, then a smaller FP8 call over what the wide one left."""
    f8 = W.make_host_inputs(W.small_shape(
        "na3", batch=4, q_len=2, num_q_heads=8, num_kv_heads=2, lo=300, hi=2500,
        paged=True, causal=True, seed=93, kv_fp8=True))
    wide = W.make_host_inputs(W.small_shape(
        "na4", batch=3, q_len=8, num_q_heads=16, num_kv_heads=2, lo=300, hi=2500,
        paged=True, causal=True, seed=94))
    f8_small = W.make_host_inputs(W.small_shape(
        "na5", batch=2, q_len=1, num_q_heads=4, num_kv_heads=2, lo=400, hi=700,
        paged=True, seed=95, kv_fp8=True))
    check_pair(binding, ((f8, 5), (wide, 4), (f8_small, 2)))


def test_oversized_call_is_rejected_without_launch(binding):
    # 256 x 64 rows x 64 splits x 516 B of partials >> 16 MiB
    p = binding.decode_attn_params_init(256, 1, 64, 8, 128, 0, 0, 0, 32768, False)
    assert binding.decode_attn_workspace_bytes(p, 64) > binding.STATIC_WORKSPACE_BYTES
    rc = binding.lib().decode_attn_static_workspace(ctypes.byref(p), None, None, None, None,
                                                    None, None, None, 64, None, None)
    assert rc == binding.DA_ERR_STATIC_WORKSPACE_LIMIT
    assert "16 MiB" in binding.decode_attn_status_string(rc)
