"""GPU parity of the CUDA path against the fp64 oracle (small and ragged cases).

Every call goes through the C ABI (ctypes binding).  Sizes span several
16-token tiles, several 64-token pipeline stages and several chunks, with
ragged tails; the tolerance rule is in tests/parity.py.
"""
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


def run(binding, inp, num_splits=0, status=None, **kw):
    q, k, v, bt, lens = to_device(inp)
    out, lse = binding.decode_attn(q, k, v, bt, lens, max_seq_len=inp.max_seq_len,
                                   causal=inp.shape.causal, scale=inp.shape.scale,
                                   num_splits=num_splits, status=status,
                                   k_scale=inp.k_scale, v_scale=inp.v_scale, **kw)
    torch.cuda.synchronize()
    return out, lse


def check(binding, inp, num_splits=0, two_pass=False):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(binding, inp, num_splits, status=status, two_pass=two_pass)
    ref_o, ref_l = oracle.decode_attention_inputs(inp)
    assert int(status.item()) == 0
    assert_out_close(bf16_tensor_to_f64(out), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)
    assert_ulps_close(bf16_tensor_to_bits(out), ref_o)
    return out, lse


CASES = [
    # name, G, q_len, causal, paged, page_size, lo, hi
    ("mha_contig", 1, 1, False, False, 16, 1, 700),
    ("gqa4_paged", 4, 1, False, True, 16, 1, 900),
    ("gqa8_paged_peaked", 8, 1, False, True, 16, 100, 1200),
    ("gqa4_q4_causal", 4, 4, True, True, 16, 4, 800),
    ("gqa4_q4_nocausal", 4, 4, False, True, 16, 4, 600),
    ("gqa2_q3_causal_contig", 2, 3, True, False, 16, 3, 500),
    ("gqa16_paged", 16, 1, False, True, 16, 1, 400),
    ("mha_q16_causal", 1, 16, True, True, 16, 16, 300),
    ("gqa4_q2_page32", 4, 2, True, True, 32, 2, 700),
    ("gqa8_page64", 8, 1, False, True, 64, 1, 500),
    # wide query groups (17..128 rows per kv head): the tcgen05 kernel
    ("wide20_gqa4_q5_causal_contig", 4, 5, True, False, 16, 5, 600),
    ("wide32_gqa8_q4_causal", 8, 4, True, True, 16, 4, 900),
    ("wide64_gqa8_q8_causal", 8, 8, True, True, 16, 8, 700),
    ("wide64_gqa16_q4_nocausal_page32", 16, 4, False, True, 32, 4, 500),
    ("wide128_gqa16_q8_causal", 16, 8, True, True, 16, 8, 400),
    ("wide128_mha_q128_causal", 1, 128, True, True, 16, 128, 400),
]


@pytest.mark.parametrize("two_pass", [False, True], ids=["merge-auto", "two-pass"])
@pytest.mark.parametrize("splits", [1, 2, 7, 0])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_small_workloads_match_oracle(binding, case, splits, two_pass):
    name, G, T, causal, paged, ps, lo, hi = case
    shp = W.small_shape(name, batch=4, q_len=T, num_q_heads=2 * G, num_kv_heads=2,
                        lo=lo, hi=hi, paged=paged, page_size=ps, causal=causal,
                        peaked=0.05 if "peaked" in name else 0.0, seed=100 + G + T)
    inp = W.make_host_inputs(shp)
    check(binding, inp, splits, two_pass)


@pytest.mark.parametrize("splits", [1, 3])
def test_edge_lengths_including_empty_requests(binding, splits):
    lens = np.array([0, 1, 15, 16, 17, 63, 64, 65, 127, 129, 0, 250], np.int32)
    shp = W.small_shape("edges", batch=len(lens), num_q_heads=8, num_kv_heads=2,
                        lo=0, hi=256, paged=True, seed=31)
    inp = W.make_host_inputs(shp, seq_lens=lens)
    out, lse = check(binding, inp, splits)
    o = bf16_tensor_to_f64(out)
    assert np.all(o[0] == 0) and np.all(o[10] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[[0, 10]]))


@pytest.mark.parametrize("splits", [1, 3])
def test_wide_edge_lengths_including_empty_requests(binding, splits):
    lens = np.array([0, 4, 15, 16, 17, 63, 64, 65, 127, 129, 0, 250], np.int32)
    shp = W.small_shape("wide_edges", batch=len(lens), q_len=4, num_q_heads=16,
                        num_kv_heads=2, lo=0, hi=256, paged=True, causal=True, seed=35)
    inp = W.make_host_inputs(shp, seq_lens=lens)
    out, lse = check(binding, inp, splits)
    assert np.all(bf16_tensor_to_f64(out)[[0, 10]] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[[0, 10]]))


@pytest.mark.parametrize("direction", [1.0, -1.0])
def test_wide_running_max_keeps_moving(binding, direction):
    """Scores that drift steadily up (or down) along the sequence make the
    running max grow by more than 2^8 many times within one chunk, so the
    tcgen05 kernel's lazy O rescaling runs repeatedly."""
    rng = np.random.default_rng(36)
    B, T, Hq, Hkv, L = 2, 8, 64, 4, 1500
    q = rng.standard_normal((B, T, Hq, 128)).astype(np.float32)
    k = rng.standard_normal((B, L, Hkv, 128)).astype(np.float32) * 0.3
    # add a component along the mean query direction that grows with j
    qdir = q.reshape(B, T, Hkv, Hq // Hkv, 128).mean(axis=(1, 3))          # [B, Hkv, 128]
    qdir /= np.linalg.norm(qdir, axis=-1, keepdims=True)
    ramp = direction * np.linspace(0, 60, L, dtype=np.float32)              # scale x ramp >> 2^8
    k += ramp[None, :, None, None] * qdir[:, None, :, :]
    v = rng.standard_normal((B, L, Hkv, 128)).astype(np.float32)
    inp = W.DecodeInputs(W.small_shape("ramp", batch=B, q_len=T, num_q_heads=Hq,
                                       num_kv_heads=Hkv, lo=L, hi=L, paged=False, causal=True),
                         W.f32_to_bf16_bits(q), W.f32_to_bf16_bits(k), W.f32_to_bf16_bits(v),
                         None, np.full(B, L, np.int32), L, 0, 0)
    for S in (1, 2):
        check(binding, inp, S)


def test_all_requests_empty(binding):
    shp = W.small_shape("empty", batch=3, num_q_heads=4, num_kv_heads=1, lo=0, hi=0,
                        paged=False, seed=32)
    inp = W.make_host_inputs(shp, seq_lens=np.zeros(3, np.int32))
    q, _, _, _, lens = to_device(inp)
    # contiguous cache with max_seq_len = 0: caches may be empty
    k = torch.empty((3, 0, 1, 128), dtype=torch.bfloat16, device="cuda")
    out, lse = binding.decode_attn(q, k, k, None, lens, max_seq_len=0, num_splits=1)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0)
    assert torch.all(torch.isneginf(lse))


def test_long_single_request_many_splits(binding):
    shp = W.small_shape("long", batch=1, num_q_heads=4, num_kv_heads=1, lo=20011,
                        hi=20011, paged=False, seed=33)
    inp = W.make_host_inputs(shp)
    for s in (1, 5, 16, 40, 0):
        check(binding, inp, s)
        check(binding, inp, s, two_pass=True)


def test_cluster_merge_is_one_launch_and_matches_two_pass(binding):
    """2..16 chunks per head that fit at once merge through a thread-block
    cluster (one launch); more chunks, or the two-pass flag, use partials and
    the combine kernel.  Both forms agree with the oracle."""
    shp = W.small_shape("cm", batch=3, q_len=2, num_q_heads=16, num_kv_heads=4, lo=100,
                        hi=4000, paged=True, causal=True, seed=34)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True)
    p2 = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True,
                                     two_pass=True)
    for S in (2, 9, 16):
        assert binding.decode_attn_launch_count(p, S) == 1
        assert binding.decode_attn_launch_count(p2, S) == 2
        o1, l1 = check(binding, inp, S)
        o2, l2 = check(binding, inp, S, two_pass=True)
        assert_out_close(bf16_tensor_to_f64(o1), bf16_tensor_to_f64(o2), what="cluster vs two-pass")
    # beyond the largest cluster (after rounding the chunk length to 16 tokens)
    assert binding.decode_attn_launch_count(p, 40) == 2


@pytest.mark.parametrize("batch", [3, 300, 1030])
def test_wide_schedule_batch_sizes(binding, batch):
    """The tcgen05 kernel's persistent schedule over batches of every kind:
    few requests (partial chunks sorted by length), more than the sorting
    limit (index order), and more than its tables hold (one item per CTA);
    lengths include empty requests, full and partial chunks."""
    rng = np.random.default_rng(40 + batch)
    lens = rng.integers(4, 200, batch).astype(np.int32)  # causal: at least q_len keys
    lens[:: 7] = 0
    lens[1:: 11] = 160  # two full 80-token chunks at 3 splits
    shp = W.small_shape("wide_sched", batch=batch, q_len=4, num_q_heads=16, num_kv_heads=2,
                        lo=0, hi=200, paged=True, causal=True, seed=41 + batch)
    inp = W.make_host_inputs(shp, seq_lens=lens)
    for S in (1, 3):
        out, lse = check(binding, inp, S)
        assert np.all(bf16_tensor_to_f64(out)[lens == 0] == 0)


@pytest.mark.parametrize("two_pass", [False, True], ids=["merge-auto", "two-pass"])
@pytest.mark.parametrize("splits", [1, 3, 7])
@pytest.mark.parametrize("G,q_len,causal", [(4, 1, False), (4, 4, True), (8, 2, True)],
                         ids=["rows4", "rows16_causal", "rows16_q2"])
def test_grids_beyond_one_wave_match_oracle(binding, G, q_len, causal, splits, two_pass):
    """Grids of more CTAs than SMs run the default pipeline shape (grids of at
    most one CTA per SM run the deeper one, which the smaller cases cover):
    40 requests x 4 kv heads x splits CTAs."""
    shp = W.small_shape("wave", batch=40, q_len=q_len, num_q_heads=4 * G, num_kv_heads=4,
                        lo=q_len, hi=300, paged=True, causal=causal, seed=50 + G + q_len)
    inp = W.make_host_inputs(shp)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 40 * 4 * splits > sms
    check(binding, inp, splits, two_pass=two_pass)


def test_plan_small_ragged_batch_fills_the_gpu(binding):
    """A small ragged batch with wide query groups: the per-row chunk floor (64
    tokens per query row) would leave far fewer chunks than the tcgen05
    kernel's CTA slots (one per SM); the planner shrinks the chunk until they
    fill one wave, and the result still matches the oracle."""
    shp = W.small_shape("plan_small", batch=2, q_len=8, num_q_heads=64, num_kv_heads=8,
                        lo=2000, hi=5000, paged=True, causal=True, seed=42)
    inp = W.make_host_inputs(shp)
    q, k, v, bt, lens = to_device(inp)
    p = binding.params_from_tensors(q, k, bt, max_seq_len=inp.max_seq_len, causal=True)
    S, chunk = binding.decode_attn_plan(p, inp.seq_lens)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chunks = sum(max(1, -(-int(L) // chunk)) for L in inp.seq_lens) * shp.num_kv_heads
    assert 256 <= chunk < 64 * 64
    assert chunks >= sms
    check(binding, inp, 0)
    check(binding, inp, S, two_pass=True)


# FP8 E4M3 caches (one scale per cache): the narrow kernel widens them to f16
FP8_CASES = [
    # name, G, q_len, causal, paged, page_size, lo, hi
    ("f8_mha_contig", 1, 1, False, False, 16, 1, 700),
    ("f8_gqa4_paged", 4, 1, False, True, 16, 1, 900),
    ("f8_gqa8_paged_peaked", 8, 1, False, True, 16, 100, 1200),
    ("f8_gqa4_q4_causal", 4, 4, True, True, 16, 4, 800),
    ("f8_gqa16_paged", 16, 1, False, True, 16, 1, 400),
    ("f8_mha_q16_causal", 1, 16, True, True, 16, 16, 300),
    ("f8_gqa4_q2_page32", 4, 2, True, True, 32, 2, 700),
    # wide query groups with FP8 caches: the tcgen05 kernel widens them to f16
    ("f8w32_gqa8_q4_causal", 8, 4, True, True, 16, 4, 900),
    ("f8w64_gqa16_q4_page32", 16, 4, False, True, 32, 4, 600),
    ("f8w128_gqa16_q8_causal", 16, 8, True, True, 16, 8, 500),
]


@pytest.mark.parametrize("two_pass", [False, True], ids=["merge-auto", "two-pass"])
@pytest.mark.parametrize("splits", [1, 2, 7, 0])
@pytest.mark.parametrize("case", FP8_CASES, ids=[c[0] for c in FP8_CASES])
def test_fp8_cache_workloads_match_oracle(binding, case, splits, two_pass):
    name, G, T, causal, paged, ps, lo, hi = case
    shp = W.small_shape(name, batch=4, q_len=T, num_q_heads=2 * G, num_kv_heads=2,
                        lo=lo, hi=hi, paged=paged, page_size=ps, causal=causal,
                        peaked=0.05 if "peaked" in name else 0.0, seed=200 + G + T,
                        kv_fp8=True)
    inp = W.make_host_inputs(shp)
    check(binding, inp, splits, two_pass)


@pytest.mark.parametrize("splits", [1, 3])
def test_fp8_edge_lengths_including_empty_requests(binding, splits):
    lens = np.array([0, 1, 15, 16, 17, 63, 64, 65, 127, 129, 0, 250], np.int32)
    shp = W.small_shape("f8_edges", batch=len(lens), num_q_heads=8, num_kv_heads=2,
                        lo=0, hi=256, paged=True, seed=37, kv_fp8=True)
    inp = W.make_host_inputs(shp, seq_lens=lens)
    out, lse = check(binding, inp, splits)
    assert np.all(bf16_tensor_to_f64(out)[[0, 10]] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[[0, 10]]))
