"""Full-size parity on the decode workloads (bf16 and FP8 caches), in the launch configuration
the benchmark times (the library planner fed the host sequence lengths).

The oracle computes a sample of output rows one by one (every row of a few
requests, plus random rows); every row is also checked for properties that
hold at any size: finite outputs, each output a convex combination of value
rows (|out| <= max |V| + tolerance), finite LSE for non-empty requests, and
a clean device status word."""
import numpy as np
import pytest

import oracle
from split_kv_decode_attention_gb300 import workloads as W
from tests.parity import (assert_lse_close, assert_out_close, assert_ulps_close,
                          bf16_tensor_to_bits, bf16_tensor_to_f64)

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from split_kv_decode_attention_gb300 import binding as B
    from split_kv_decode_attention_gb300 import build as cuda_build
    cuda_build.build()
    B.lib()
    return B


def host_bits(t):
    if t.element_size() == 1:   # FP8 E4M3 bytes
        return t.contiguous().cpu().numpy().view(np.uint8)
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER + list(W.WIDE_WORKLOADS) + list(W.FP8_WORKLOADS))
def test_full_size_workload_sampled_rows_match_oracle(binding, name):
    shape = W.WORKLOADS[name]
    inp = W.make_device_inputs(shape, device="cuda")
    lens_h = inp.seq_lens.cpu().numpy()
    q, k, v, bt, lens = inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seq_lens
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len,
                                    causal=shape.causal, scale=shape.scale,
                                    k_scale=inp.k_scale, v_scale=inp.v_scale)
    S, _ = binding.decode_attn_plan(p, lens_h)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len,
                                   causal=shape.causal, scale=shape.scale, num_splits=S,
                                   status=status, params=p)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    o = bf16_tensor_to_f64(out)
    l = lse.cpu().numpy()
    vmax = 448.0 * inp.v_scale if shape.kv_fp8 else float(v.float().abs().max().item())
    assert np.all(np.isfinite(o))
    assert np.abs(o).max() <= vmax + 1e-2
    assert np.all(np.isfinite(l[lens_h > 0]))

    # rows: all rows of the shortest and longest request, plus random rows
    B, T, Hq = shape.batch, shape.q_len, shape.num_q_heads
    rng = np.random.default_rng(7)
    whole = {int(np.argmin(lens_h)), int(np.argmax(lens_h))}
    rows = [(b * T + t) * Hq + h for b in sorted(whole) for t in range(T) for h in range(Hq)]
    rows += rng.choice(B * T * Hq, size=min(64, B * T * Hq), replace=False).tolist()
    rows = np.array(sorted(set(rows)), np.int32)
    host = W.DecodeInputs(shape, host_bits(q), host_bits(k), host_bits(v),
                          None if bt is None else bt.cpu().numpy(), lens_h,
                          inp.max_seq_len, inp.num_pages, inp.page_size, inp.k_scale,
                          inp.v_scale)
    ref_o, ref_l = oracle.decode_attention_inputs(host, rows=rows)
    assert_out_close(o.reshape(-1, 128)[rows], ref_o, what=name)
    assert_lse_close(l.reshape(-1)[rows], ref_l, what=name)
    assert_ulps_close(bf16_tensor_to_bits(out).reshape(-1, 128)[rows], ref_o, what=name)
