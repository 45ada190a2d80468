"""GPU checks of the paged gather, the split partials, the combine step, the
device status word and CUDA-graph capture.  All calls go through the C ABI."""
import zlib

import numpy as np
import pytest

import oracle
from split_kv_decode_attention_gb300 import workloads as W
from tests.parity import (assert_lse_close, assert_out_close, bf16_tensor_to_bits,
                          bf16_tensor_to_f64, to_device)
from tests.test_oracle_pins import paginate

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


def bf(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


# ---------------------------------------------------------------- paging
@pytest.mark.parametrize("splits", [1, 3])
def test_fp8_shuffled_pages_bit_identical_to_contiguous(binding, splits):
    """FP8 E4M3 caches: the same logical bytes contiguous and as shuffled
    pages give identical bits out."""
    rng = np.random.default_rng(60 + splits)
    B, Lmax, Hkv, Hq, D = 5, 1000, 2, 8, 128
    kc, ks = W.quantize_e4m3(rng.standard_normal((B, Lmax, Hkv, D), dtype=np.float32))
    vc, vs = W.quantize_e4m3(rng.standard_normal((B, Lmax, Hkv, D), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((B, 1, Hq, D), dtype=np.float32))
    lens = np.array([1000, 1, 333, 16, 777], np.int32)
    kp, vp, bt = paginate(kc, vc, lens, 16, rng)
    lens_d = torch.from_numpy(lens).cuda()
    u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    o1, l1 = binding.decode_attn(bf(q), u8(kc), u8(vc), None, lens_d, max_seq_len=Lmax,
                                 num_splits=splits, k_scale=ks, v_scale=vs)
    o2, l2 = binding.decode_attn(bf(q), u8(kp), u8(vp), torch.from_numpy(bt).cuda(), lens_d,
                                 max_seq_len=Lmax, num_splits=splits, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_to_bits(o1), bf16_tensor_to_bits(o2))
    assert np.array_equal(l1.cpu().numpy().view(np.uint32), l2.cpu().numpy().view(np.uint32))
    ref_o, ref_l = oracle.decode_attention(q, kc, vc, lens, num_kv_heads=Hkv, kv_fp8=True,
                                           k_scale=ks, v_scale=vs)
    assert_out_close(bf16_tensor_to_f64(o2), ref_o)
    assert_lse_close(l2.cpu().numpy(), ref_l)


@pytest.mark.parametrize("page_size", [16, 32, 128])
@pytest.mark.parametrize("splits", [1, 3])
def test_shuffled_pages_bit_identical_to_contiguous(binding, page_size, splits):
    """Same logical K/V stored contiguously and as shuffled pages: identical
    bits out (the reduction order depends on logical positions only)."""
    rng = np.random.default_rng(40 + page_size)
    B, Lmax, Hkv, Hq, D = 5, 1000, 2, 8, 128
    kc = W.f32_to_bf16_bits(rng.standard_normal((B, Lmax, Hkv, D), dtype=np.float32))
    vc = W.f32_to_bf16_bits(rng.standard_normal((B, Lmax, Hkv, D), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((B, 1, Hq, D), dtype=np.float32))
    lens = np.array([1000, 1, 333, 16, 777], np.int32)
    kp, vp, bt = paginate(kc, vc, lens, page_size, rng)
    lens_d = torch.from_numpy(lens).cuda()
    o1, l1 = binding.decode_attn(bf(q), bf(kc), bf(vc), None, lens_d, max_seq_len=Lmax,
                                 num_splits=splits)
    o2, l2 = binding.decode_attn(bf(q), bf(kp), bf(vp), torch.from_numpy(bt).cuda(), lens_d,
                                 max_seq_len=Lmax, num_splits=splits)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_to_bits(o1), bf16_tensor_to_bits(o2))
    assert np.array_equal(l1.cpu().numpy().view(np.uint32), l2.cpu().numpy().view(np.uint32))
    ref_o, ref_l = oracle.decode_attention(q, kc, vc, lens, num_kv_heads=Hkv)
    assert_out_close(bf16_tensor_to_f64(o2), ref_o)
    assert_lse_close(l2.cpu().numpy(), ref_l)


# Every kernel variant and merge path: (rows per KV head via heads x q_len,
# causal), splits, flags.  4 rows: the 8-row warp-MMA kernel; 16 rows (GQA 4
# x 4 causal tokens): the 16-row variant with Q in shared memory; 64 and 128
# rows: the tcgen05 kernel.  "merge" lets decode_attn pick the cluster merge
# where it applies; "two-pass" forces partials in the workspace + combine.
PAGING_VARIANTS = [
    # id, Hq, Hkv, q_len, causal, splits, two_pass
    ("rows4_direct", 8, 2, 1, False, 1, False),
    ("rows4_two_pass", 8, 2, 1, False, 3, True),
    ("rows16_merge", 8, 2, 4, True, 3, False),
    ("rows16_two_pass", 8, 2, 4, True, 5, True),
    ("rows64_tcgen05_direct", 16, 2, 8, True, 1, False),
    ("rows64_tcgen05_two_pass", 16, 2, 8, True, 3, True),
    ("rows128_tcgen05_two_pass", 16, 1, 8, True, 2, True),
]


@pytest.mark.parametrize("kv_fp8", [False, True], ids=["bf16", "fp8"])
@pytest.mark.parametrize("variant", PAGING_VARIANTS, ids=[v[0] for v in PAGING_VARIANTS])
def test_every_kernel_path_bit_identical_paged_vs_contiguous(binding, variant, kv_fp8):
    """The same logical K/V stored contiguously and as shuffled 16-token
    pages give identical bits out (out and LSE) on every kernel variant and
    merge path, bf16 and FP8 caches: the gather maps logical positions
    exactly, and no reduction order depends on the physical layout."""
    name, Hq, Hkv, T, causal, splits, two_pass = variant
    rng = np.random.default_rng(zlib.crc32(name.encode()) + int(kv_fp8))
    B, Lmax, D = 5, 1100, 128
    x = lambda: rng.standard_normal((B, Lmax, Hkv, D), dtype=np.float32)  # noqa: E731
    if kv_fp8:
        (kc, ks), (vc, vs) = W.quantize_e4m3(x()), W.quantize_e4m3(x())
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    else:
        kc, vc, ks, vs = W.f32_to_bf16_bits(x()), W.f32_to_bf16_bits(x()), 1.0, 1.0
        dev = bf
    q = W.f32_to_bf16_bits(rng.standard_normal((B, T, Hq, D), dtype=np.float32))
    lens = np.array([1100, T, 333, 16 + T, 777], np.int32)
    kp, vp, bt = paginate(kc, vc, lens, 16, rng)
    lens_d = torch.from_numpy(lens).cuda()
    kw = dict(max_seq_len=Lmax, num_splits=splits, causal=causal, two_pass=two_pass,
              k_scale=ks, v_scale=vs)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o1, l1 = binding.decode_attn(bf(q), dev(kc), dev(vc), None, lens_d, status=status, **kw)
    o2, l2 = binding.decode_attn(bf(q), dev(kp), dev(vp), torch.from_numpy(bt).cuda(), lens_d,
                                 status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bf16_tensor_to_bits(o1), bf16_tensor_to_bits(o2))
    assert np.array_equal(l1.cpu().numpy().view(np.uint32), l2.cpu().numpy().view(np.uint32))
    ref_o, ref_l = oracle.decode_attention(q, kc, vc, lens, num_kv_heads=Hkv, causal=causal,
                                           kv_fp8=kv_fp8, k_scale=ks, v_scale=vs)
    assert_out_close(bf16_tensor_to_f64(o2), ref_o)
    assert_lse_close(l2.cpu().numpy(), ref_l)


def test_strided_head_major_cache_matches_oracle(binding):
    """Caches laid out [page, head, slot, d] (head outer) through the strides."""
    shp = W.small_shape("hm", batch=3, num_q_heads=8, num_kv_heads=2, lo=30, hi=300, seed=41)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    k_hm = k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)   # same shape, new strides
    v_hm = v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert k_hm.stride() != k.stride()
    out, lse = binding.decode_attn(q, k_hm, v_hm, bt, lens, max_seq_len=inp.max_seq_len,
                                   num_splits=2)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)


# ---------------------------------------------------------------- partials
def test_split_partials_match_oracle_on_each_chunk(binding):
    shp = W.small_shape("parts", batch=3, q_len=2, num_q_heads=8, num_kv_heads=2, lo=200,
                        hi=900, causal=True, seed=42)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True,
                                    two_pass=True)       # partials are only kept in two passes
    S = 4
    chunk = binding.decode_attn_chunk_len(p, S)
    ws = torch.full(((binding.decode_attn_workspace_bytes(p, S) + 3) // 4,), float("nan"),
                    dtype=torch.float32, device="cuda")
    binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, causal=True,
                        num_splits=S, workspace=ws, params=p)
    torch.cuda.synchronize()
    po, pl = binding.workspace_views(ws, p, S)
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    for b in range(shp.batch):
        nb = max(1, -(-int(inp.seq_lens[b]) // chunk))
        if nb < 2:
            continue
        rows = np.arange(b * 2 * 8, (b + 1) * 2 * 8, dtype=np.int32)
        for s in range(nb):
            ro, rl = oracle.decode_attention_inputs(inp, rows=rows, key_lo=s * chunk,
                                                    key_hi=(s + 1) * chunk)
            assert_out_close(po[b, :, :, s].reshape(-1, 128), ro, what=f"partial b{b} s{s}")
            assert_lse_close(pl[b, :, :, s].reshape(-1), rl, what=f"partial lse b{b} s{s}")


def test_combine_alone_matches_oracle_merge(binding):
    rng = np.random.default_rng(43)
    B, T, Hq, S, chunk = 3, 2, 4, 6, 64
    lens = np.array([S * chunk, 2 * chunk - 5, chunk], np.int32)   # 6, 2 and 1 chunks
    p = binding.decode_attn_params_init(B, T, Hq, 1, 128, 0, 0, 0, S * chunk, False)
    p.flags = binding.DA_FLAG_TWO_PASS       # the workspace holds partials to merge
    part_o = rng.standard_normal((B, T, Hq, S, 128)).astype(np.float32)
    part_l = (rng.standard_normal((B, T, Hq, S)) * 5).astype(np.float32)
    part_l[0, 0, 0, 2] = -np.inf
    part_o[0, 0, 0, 2] = 0
    part_l[1, 1, 3, :] = -np.inf                                     # a row with no keys
    part_o[1, 1, 3, :] = 0
    ws = torch.from_numpy(np.concatenate([part_o.ravel(), part_l.ravel()])).cuda()
    out = torch.full((B, T, Hq, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, T, Hq), 7.0, dtype=torch.float32, device="cuda")
    binding.decode_attn_combine(p, torch.from_numpy(lens).cuda(), S, chunk, ws, out, lse)
    torch.cuda.synchronize()
    nvalid = np.array([6, 2, 1])[:, None, None] * np.ones((1, T, Hq), int)
    ref_o, ref_l = oracle.merge_partials(part_o.astype(np.float64), part_l.astype(np.float64),
                                         nvalid=nvalid)
    o = bf16_tensor_to_f64(out)
    assert_out_close(o[:2], ref_o[:2])
    assert_lse_close(lse.cpu().numpy()[:2], ref_l[:2])
    # the single-chunk request is the split kernel's to write: untouched here
    assert torch.all(out[2].float() == 7.0) and torch.all(lse[2] == 7.0)


# ---------------------------------------------------------------- status word
def test_bad_page_entry_sets_status_and_does_not_fault(binding):
    shp = W.small_shape("badpage", batch=4, num_q_heads=8, num_kv_heads=2, lo=40, hi=200,
                        seed=44)
    inp = W.make_host_inputs(shp)
    bt = inp.block_table.copy()
    bt[1, 0] = inp.num_pages + 5
    bt[2, 1] = -3
    q, k, v, _, lens = to_device(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.decode_attn(q, k, v, torch.from_numpy(bt).cuda(), lens,
                                   max_seq_len=inp.max_seq_len, num_splits=2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.DA_STATUS_BAD_PAGE
    # untouched requests are still exact
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    o = bf16_tensor_to_f64(out)
    for b in (0, 3):
        assert_out_close(o[b], ref_o[b])
        assert_lse_close(lse.cpu().numpy()[b], ref_l[b])


def test_seq_len_beyond_max_is_clamped_and_reported(binding):
    shp = W.small_shape("toolong", batch=2, num_q_heads=4, num_kv_heads=1, lo=100, hi=100,
                        paged=False, seed=45)
    inp = W.make_host_inputs(shp)
    q, k, v, _, _ = to_device(inp)
    lens = torch.tensor([100, 150], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.decode_attn(q, k, v, None, lens, max_seq_len=100, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == binding.DA_STATUS_SEQ_LEN
    ref_o, ref_l = oracle.decode_attention_inputs(inp)       # both requests at 100
    assert_out_close(bf16_tensor_to_f64(out), ref_o)


def test_short_causal_request_is_reported(binding):
    shp = W.small_shape("short", batch=2, q_len=4, num_q_heads=8, num_kv_heads=2, lo=2, hi=2,
                        causal=True, seed=46)
    inp = W.make_host_inputs(shp, seq_lens=np.array([2, 50], np.int32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v, bt, lens = to_device(inp)
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=50, causal=True,
                                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == binding.DA_STATUS_SHORT_CAUSAL
    ref_o, ref_l = oracle.decode_attention_inputs(inp)       # rows with no key: 0 / -inf
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)


def test_workspace_too_small_is_rejected(binding):
    shp = W.small_shape("ws", batch=2, num_q_heads=4, num_kv_heads=1, lo=500, hi=500,
                        paged=False, seed=47)
    q, k, v, _, lens = to_device(W.make_host_inputs(shp))
    p = binding.params_from_tensors(q, k, None, max_seq_len=500, two_pass=True)
    need = binding.decode_attn_workspace_bytes(p, 4)
    ws = torch.empty(need // 4 - 1, dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    import ctypes
    rc = binding.lib().decode_attn(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   None, lens.data_ptr(), out.data_ptr(), lse.data_ptr(), 4,
                                   ws.data_ptr(), ws.numel() * 4, None, None)
    assert rc == -7


# ---------------------------------------------------------------- graph capture
def test_call_replays_inside_a_cuda_graph(binding):
    shp = W.small_shape("graph", batch=4, num_q_heads=16, num_kv_heads=2, lo=100, hi=3000,
                        seed=48)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len)
    S = 5
    ws = torch.empty((binding.decode_attn_workspace_bytes(p, S) + 3) // 4,
                     dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, num_splits=S,
                            out=out, lse=lse, workspace=ws, params=p, stream=s)   # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, num_splits=S,
                            out=out, lse=lse, workspace=ws, params=p, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)



@pytest.mark.parametrize("kind", ["wide", "fp8", "fp8_wide"])
def test_wide_and_fp8_calls_replay_inside_a_cuda_graph(binding, kind):
    """The persistent tcgen05 kernel (64 rows per KV head) and the FP8-cache
    paths captured in a CUDA graph and replayed."""
    if kind in ("wide", "fp8_wide"):
        shp = W.small_shape("graph_w", batch=5, q_len=8, num_q_heads=16, num_kv_heads=2,
                            lo=100, hi=3000, causal=True, seed=49, kv_fp8=kind == "fp8_wide")
    else:
        shp = W.small_shape("graph_f8", batch=4, q_len=2, num_q_heads=8, num_kv_heads=2,
                            lo=100, hi=3000, causal=True, seed=50, kv_fp8=True)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True,
                                    k_scale=inp.k_scale, v_scale=inp.v_scale)
    S = 3
    ws = torch.empty((binding.decode_attn_workspace_bytes(p, S) + 3) // 4 + 1,
                     dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, num_splits=S,
                            out=out, lse=lse, workspace=ws, params=p, stream=s)   # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, num_splits=S,
                            out=out, lse=lse, workspace=ws, params=p, stream=s)
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)



def test_withheld_copy_times_out_and_context_stays_usable(binding):
    """Failure detection without a GPU fault: the test flag makes block
    (0, 0, 0) of the split launch withhold its first pipeline stage, so that
    block's bounded wait runs out (~2 s) and the call reports
    DA_STATUS_TIMEOUT; the next call on the same context is exact."""
    import time
    shp = W.small_shape("withhold", batch=2, num_q_heads=8, num_kv_heads=2, lo=500, hi=900,
                        seed=70)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, two_pass=True)
    p.flags |= binding.DA_FLAG_TEST_WITHHOLD_COPY
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, num_splits=2,
                        status=status, params=p)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.DA_STATUS_TIMEOUT
    assert time.time() - t0 < 60
    status.zero_()
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len,
                                   num_splits=2, status=status, two_pass=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)


def test_withheld_copy_times_out_in_the_tcgen05_kernel_and_context_stays_usable(binding):
    """The same failure detection on the tcgen05 kernel (64 rows per KV head):
    CTA 0 never fills the first stage of its first work item, so the MMA
    warp's idle limit and the softmax warps' bounded waits run out, the
    groups' statistics exchange and the TMEM release wait on bounded
    mbarriers, and the call reports DA_STATUS_TIMEOUT; the next call on the
    same context is exact."""
    import time
    shp = W.small_shape("withhold_wide", batch=2, q_len=8, num_q_heads=16, num_kv_heads=2,
                        lo=500, hi=900, causal=True, seed=71)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True,
                                    two_pass=True)
    p.flags |= binding.DA_FLAG_TEST_WITHHOLD_COPY
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, causal=True,
                        num_splits=2, status=status, params=p)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.DA_STATUS_TIMEOUT
    assert time.time() - t0 < 60
    status.zero_()
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len, causal=True,
                                   num_splits=2, status=status, two_pass=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)


def test_withheld_copy_times_out_in_the_fp8_tcgen05_kernel_and_context_stays_usable(binding):
    """The same on the tcgen05 kernel's FP8 variant, whose converter warps
    wait on the TMA stage and on free K and V operand slots: CTA 0's first
    stage never lands, so the converters' bounded waits run out, the MMA
    warp's idle limit runs out waiting for widened K, and the call reports
    DA_STATUS_TIMEOUT; the next call on the same context is exact."""
    import time
    shp = W.small_shape("withhold_wide_fp8", batch=2, q_len=8, num_q_heads=16, num_kv_heads=2,
                        lo=500, hi=900, causal=True, seed=72, kv_fp8=True)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    kw = dict(max_seq_len=inp.max_seq_len, causal=True, k_scale=inp.k_scale,
              v_scale=inp.v_scale)
    p = binding.params_from_tensors(q, k, bt, two_pass=True, **kw)
    p.flags |= binding.DA_FLAG_TEST_WITHHOLD_COPY
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    binding.decode_attn(q, k, v, bt, lens, num_splits=2, status=status, params=p,
                        max_seq_len=inp.max_seq_len, causal=True)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.DA_STATUS_TIMEOUT
    assert time.time() - t0 < 60
    status.zero_()
    out, lse = binding.decode_attn(q, k, v, bt, lens, num_splits=2, status=status,
                                   two_pass=True, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)
