"""Device planning: decode_attn(num_splits <= 0) with two or more requests
plans on the GPU from the lengths in device memory (a planner kernel before
the split launch), so the call stays graph-capturable and a replay plans for
the lengths current at replay time.  Checked through the C ABI: the device
plan equals the host planner's plan for the same lengths, the item list and
prefixes are what they should be, outputs match the fp64 oracle and are bit
identical to the explicit host plan, and a captured graph re-plans when the
lengths change between replays."""
import dataclasses

import numpy as np
import pytest

import oracle
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


def plan_params(binding, batch, q_len, hq, hkv, max_seq_len, page_size=16, causal=False,
                fp8=False):
    max_pages = max(1, -(-max_seq_len // page_size)) if page_size else 0
    p = binding.decode_attn_params_init(batch, q_len, hq, hkv, 128, page_size, max_pages,
                                        max(1, batch * max_pages), max_seq_len, causal)
    if fp8:
        p.flags |= binding.DA_FLAG_KV_FP8_E4M3
    return p


def device_plan(binding, p, lens):
    ws = torch.zeros((binding.decode_attn_workspace_bytes(p, 0) + 3) // 4, dtype=torch.int32,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.decode_attn_device_plan(p, torch.from_numpy(np.asarray(lens, np.int32)).cuda(), ws,
                                    status=status)
    torch.cuda.synchronize()
    plan, pre, items = binding.device_plan_view(ws, p)
    return (plan.cpu().numpy(), pre.cpu().numpy(), items.cpu().numpy(), int(status.item()))


def check_plan(binding, p, lens):
    lens = np.asarray(lens, np.int32)
    plan, pre, items, st = device_plan(binding, p, lens)
    S, chunk = binding.decode_attn_plan(p, lens)
    assert (int(plan[0]), int(plan[2])) == (chunk, S), (plan, S, chunk)
    L = np.clip(lens.astype(np.int64), 0, p.max_seq_len)
    n = np.where(L > 0, -(-L // chunk), 1)
    assert int(plan[1]) == int(n.sum()) * p.num_kv_heads <= int(plan[3])
    np.testing.assert_array_equal(pre, np.concatenate([[0], np.cumsum(n)]))
    want = np.array([(b, h, s, L[b]) for b in range(len(L)) for h in range(p.num_kv_heads)
                     for s in range(n[b])], np.int64).reshape(-1, 4)
    np.testing.assert_array_equal(items[:int(plan[1])].astype(np.int64), want)
    return plan, st


BENCH = ["c3_b64_h32kv8_L512-32768_paged", "c4_b256_h64kv8_L128-4096_paged_peaked",
         "c5_b32_q4_causal_h32kv8_L1024-16384_paged",
         "f5_b32_q4_causal_h32kv8_L1024-16384_paged_fp8",
         "w64_b32_q8_h64kv8_causal_L1024-16384_paged",
         "w128_b16_q16_h64kv8_causal_L1024-16384_paged",
         "fw64_b32_q8_h64kv8_causal_L1024-16384_paged_fp8"]


@pytest.mark.parametrize("name", BENCH)
def test_device_plan_equals_host_plan_on_benchmark_lengths(binding, name):
    shp = W.WORKLOADS[name]
    lens = W.draw_seq_lens(shp, np.random.default_rng(shp.seed))
    p = plan_params(binding, shp.batch, shp.q_len, shp.num_q_heads, shp.num_kv_heads,
                    int(lens.max()), shp.page_size, shp.causal, shp.kv_fp8)
    check_plan(binding, p, lens)


@pytest.mark.parametrize("lens,q_len,hq,hkv", [
    ([11700, 15700], 8, 64, 8),                 # wide: the chunk shrinks to fill the GPU
    ([9000, 16000, 12000, 14000], 16, 64, 8),
    ([4096] * 6, 1, 32, 8),                     # equal lengths: one wave of <= 16 chunks
    ([65536, 65536], 1, 8, 8),
    ([0, 0, 0], 1, 8, 2),                       # empty requests
    ([1, 300, 0, 17, 5000], 4, 16, 4),
    (list(range(1, 3000, 7)), 1, 4, 1),         # 429 requests
    (list(np.random.default_rng(3).integers(1, 4097, 5000)), 1, 8, 8),  # beyond the smem cache
    # 24000 (request, kv head) pairs: every planner CTA writes several blocks
    (list(np.random.default_rng(4).integers(1, 4097, 3000)), 1, 8, 8),
    # 120 requests on one kv head (fewer pairs than tcgen05 CTAs): the split
    # search runs with 16 threads testing each candidate
    (list(np.random.default_rng(5).integers(1, 12000, 120)), 1, 128, 1),
    # 16 rows on one kv head, short requests: the chunks at the per-row floor
    # do not fill the CTAs, so the search runs -- 256 requests (a warp per
    # candidate) and 257 (the bisection with block sums)
    (list(np.random.default_rng(6).integers(4, 2000, 256)), 4, 4, 1),
    (list(np.random.default_rng(7).integers(4, 2000, 257)), 4, 4, 1),
])
def test_device_plan_equals_host_plan_on_shapes(binding, lens, q_len, hq, hkv):
    lens = np.asarray(lens, np.int32)
    p = plan_params(binding, len(lens), q_len, hq, hkv, max(16, int(lens.max())),
                    causal=q_len > 1)
    check_plan(binding, p, lens)


def test_planner_reports_bad_lengths(binding):
    p = plan_params(binding, 3, 4, 8, 2, 1000, causal=True)
    *_, st = device_plan(binding, p, [2000, 2, 500])    # clamped; 0 < 2 < q_len
    assert st == binding.DA_STATUS_SEQ_LEN | binding.DA_STATUS_SHORT_CAUSAL


# (name, q_len, Hq, Hkv, causal, paged, page, lo, hi, fp8): 4 / 16 rows on the
# warp-MMA kernel, 32 / 64 / 128 rows on the tcgen05 kernel
AUTO_CASES = [
    ("rows4_paged", 1, 8, 2, False, True, 16, 0, 3000, False),
    ("rows1_mha_contig", 1, 4, 4, False, False, 16, 1, 2500, False),
    ("rows16_causal", 4, 8, 2, True, True, 16, 4, 3000, False),
    ("rows8_fp8", 1, 16, 2, False, True, 32, 1, 3000, True),
    ("rows16_fp8_causal", 2, 16, 2, True, True, 16, 2, 2500, True),
    ("rows32_tcgen05", 4, 16, 2, True, True, 16, 4, 2500, False),
    ("rows64_tcgen05_fp8", 8, 16, 2, True, True, 16, 8, 2500, True),
    ("rows128_tcgen05", 8, 16, 1, True, True, 16, 8, 1500, False),
]


def run_auto(binding, inp, **kw):
    q, k, v, bt, lens = to_device(inp)
    s = inp.shape
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len,
                                   causal=s.causal, scale=s.scale, status=status,
                                   k_scale=inp.k_scale, v_scale=inp.v_scale, **kw)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


@pytest.mark.parametrize("case", AUTO_CASES, ids=[c[0] for c in AUTO_CASES])
def test_device_planned_call_matches_oracle_and_host_plan_bits(binding, case):
    name, T, hq, hkv, causal, paged, ps, lo, hi, fp8 = case
    shp = W.small_shape(name, batch=7, q_len=T, num_q_heads=hq, num_kv_heads=hkv, lo=lo, hi=hi,
                        paged=paged, page_size=ps, causal=causal, seed=500 + len(name),
                        kv_fp8=fp8)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=causal,
                                    k_scale=inp.k_scale, v_scale=inp.v_scale)
    assert binding.decode_attn_launch_count(p, 0) == 3      # planner, split, combine
    out, lse, st = run_auto(binding, inp, num_splits=0)
    assert st == 0
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)
    # the same plan made on the host and run as an explicit two-pass call:
    # identical bits (same chunks, same kernels, same merge order)
    S, _ = binding.decode_attn_plan(p, inp.seq_lens)
    out2, lse2, st2 = run_auto(binding, inp, num_splits=S, two_pass=True)
    assert st2 == 0
    assert np.array_equal(bf16_tensor_to_bits(out), bf16_tensor_to_bits(out2))
    assert np.array_equal(lse.cpu().numpy().view(np.uint32), lse2.cpu().numpy().view(np.uint32))


def test_split_and_combine_entries_run_the_device_plan(binding):
    shp = W.small_shape("sc", batch=5, q_len=2, num_q_heads=8, num_kv_heads=2, lo=1, hi=3000,
                        causal=True, seed=77)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True)
    ws = torch.empty((binding.decode_attn_workspace_bytes(p, 0) + 3) // 4, dtype=torch.float32,
                     device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    binding.decode_attn_split(p, q, k, v, bt, lens, out, lse, 0, workspace=ws)
    binding.decode_attn_combine(p, lens, 0, 0, ws, out, lse)
    ref_out, ref_lse, _ = run_auto(binding, inp, num_splits=0)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_to_bits(out), bf16_tensor_to_bits(ref_out))
    assert np.array_equal(lse.cpu().numpy().view(np.uint32), ref_lse.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("wide", [False, True], ids=["warp_mma", "tcgen05"])
def test_captured_graph_replans_when_lengths_change(binding, wide):
    """One capture of decode_attn(num_splits=0); between replays the lengths
    change in device memory (a serving loop's next step).  Every replay
    matches the oracle for the lengths current at that replay, and the plan
    it used is the host plan for them."""
    # (16 kv heads on the warp-MMA kernel: equal lengths then take 6 chunks of
    # 672 tokens, ragged ones the per-row floor, so the plans differ)
    T, hq, hkv = (8, 16, 2) if wide else (1, 16, 16)
    cap = 4000
    shp = W.small_shape("graph_auto", batch=6, q_len=T, num_q_heads=hq, num_kv_heads=hkv,
                        lo=cap, hi=cap, causal=T > 1, seed=81 + int(wide))
    full = W.make_host_inputs(shp)                  # every request holds `cap` tokens
    q, k, v, bt, lens = to_device(full)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=cap, causal=T > 1)
    ws = torch.empty((binding.decode_attn_workspace_bytes(p, 0) + 3) // 4, dtype=torch.float32,
                     device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    call = dict(max_seq_len=cap, num_splits=0, out=out, lse=lse, workspace=ws, params=p,
                status=status, stream=s)
    with torch.cuda.stream(s):
        binding.decode_attn(q, k, v, bt, lens, **call)      # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.decode_attn(q, k, v, bt, lens, **call)
    rng = np.random.default_rng(5)
    plans = set()
    for step_lens in ([cap] * 6, rng.integers(T, cap + 1, 6), [T, cap, 17 + T, 0, 999, 2048],
                      rng.integers(T, 300, 6)):
        step_lens = np.asarray(step_lens, np.int32)
        lens.copy_(torch.from_numpy(step_lens))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        inp = dataclasses.replace(full, seq_lens=step_lens)
        ref_o, ref_l = oracle.decode_attention_inputs(inp)
        assert_out_close(bf16_tensor_to_f64(out), ref_o)
        assert_lse_close(lse.cpu().numpy(), ref_l)
        plan, _, _ = binding.device_plan_view(ws, p)
        S, chunk = binding.decode_attn_plan(p, step_lens)
        assert (int(plan[0].item()), int(plan[2].item())) == (chunk, S)
        plans.add(int(plan[0].item()))
    assert len(plans) >= 2          # the replays really planned differently


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
def test_device_plan_with_more_than_32_chunks_per_request(binding, fp8):
    """A small ragged batch whose long request the planner cuts into > 32
    chunks (the combine's multi-group path), called twice on one workspace:
    identical bits both times and to the explicit two-pass call with the
    host's plan, and the oracle's result."""
    lens = np.array([30000, 100, 0, 4097, 16], np.int32)
    shp = W.small_shape("many_chunks", batch=len(lens), q_len=2, num_q_heads=8, num_kv_heads=2,
                        lo=1, hi=30000, causal=True, seed=18, kv_fp8=fp8)
    inp = W.make_host_inputs(shp, seq_lens=np.maximum(lens, 2))
    inp.seq_lens[2] = 0                               # an empty request
    q, k, v, bt, lens_d = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True,
                                    k_scale=inp.k_scale, v_scale=inp.v_scale)
    ws = torch.empty((binding.decode_attn_workspace_bytes(p, 0) + 3) // 4, dtype=torch.float32,
                     device="cuda")
    outs = []
    for splits in (0, 0, binding.decode_attn_plan(p, inp.seq_lens)[0]):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = binding.decode_attn(q, k, v, bt, lens_d, max_seq_len=inp.max_seq_len,
                                       num_splits=splits, workspace=ws if splits == 0 else None,
                                       status=status, causal=True, two_pass=splits > 0,
                                       k_scale=inp.k_scale, v_scale=inp.v_scale)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append((bf16_tensor_to_bits(out), lse.cpu().numpy().view(np.uint32)))
        if splits == 0:
            plan, _, _ = binding.device_plan_view(ws, p)
            assert int(plan[2].item()) > 32           # the long request's chunks
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    out_f = torch.from_numpy(outs[0][0].view(np.int16)).view(torch.bfloat16).float().numpy()
    assert_out_close(out_f.astype(np.float64), ref_o)
    assert_lse_close(outs[0][1].view(np.float32), ref_l)
