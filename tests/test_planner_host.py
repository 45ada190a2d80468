"""The split planner as host logic (no GPU): decode_attn_plan_slots with the
resident-CTA counts of GB300 (152 SMs; 4 resident CTAs per SM for the
warp-MMA kernel at <= 16 query rows per kv head, 1 for the tcgen05 kernel
above), checked against its stated rules and against the plans the benchmark
printed on GB300 for every workload."""
import numpy as np
import pytest

from split_kv_decode_attention_gb300 import binding
from split_kv_decode_attention_gb300 import build as cuda_build
from split_kv_decode_attention_gb300 import workloads as W

NARROW_SLOTS = 152 * 4
WIDE_SLOTS = 152 * 1

# (num_splits, chunk_len) that bench.py reported on GB300 for each workload
BENCH_PLANS = {
    "c1_b1_h32kv8_L4096": (16, 256),
    "c2_b1_mha32_L131072": (16, 8192),
    "c3_b64_h32kv8_L512-32768_paged": (19, 1680),
    "c4_b256_h64kv8_L128-4096_paged_peaked": (5, 832),
    "c5_b32_q4_causal_h32kv8_L1024-16384_paged": (16, 1024),
    "f2_b1_mha32_L131072_fp8": (16, 8192),
    "f5_b32_q4_causal_h32kv8_L1024-16384_paged_fp8": (16, 976),
    "w64_b32_q8_h64kv8_causal_L1024-16384_paged": (1, 16144),
    "w128_b16_q16_h64kv8_causal_L1024-16384_paged": (2, 7392),
    "fw64_b32_q8_h64kv8_causal_L1024-16384_paged_fp8": (1, 16256),
}


@pytest.fixture(scope="module", autouse=True)
def lib():
    cuda_build.build()
    return binding.lib()


def params(batch, q_len, hq, hkv, max_seq_len, page_size=16, causal=False):
    p = binding.DecodeAttnParams()
    max_pages = max(1, -(-max_seq_len // page_size)) if page_size else 0
    binding.lib().decode_attn_params_init(p, batch, q_len, hq, hkv, 128, page_size, max_pages,
                                          max(1, batch * max_pages), max_seq_len,
                                          1 if causal else 0)
    return p


def rows(hq, hkv, q_len):
    return hq // hkv * q_len


def slots_for(r):
    return WIDE_SLOTS if r > 16 else NARROW_SLOTS


def chunks(lens, chunk, hkv):
    lens = np.asarray(lens, np.int64)
    return int(np.sum(np.where(lens > 0, -(-lens // chunk), 1))) * hkv


@pytest.mark.parametrize("name", sorted(BENCH_PLANS))
def test_benchmark_workload_plans(name):
    shp = W.WORKLOADS[name]
    lens = W.draw_seq_lens(shp, np.random.default_rng(shp.seed))
    msl = int(lens.max())
    p = params(shp.batch, shp.q_len, shp.num_q_heads, shp.num_kv_heads, msl,
               shp.page_size if shp.paged else 0, shp.causal)
    r = rows(shp.num_q_heads, shp.num_kv_heads, shp.q_len)
    assert binding.decode_attn_plan_slots(p, lens, slots_for(r)) == BENCH_PLANS[name]


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(BENCH_PLANS))
def test_device_planner_matches_the_host_model_on_gb300(name):
    """decode_attn_plan (SM count and kernel occupancy read from the device)
    gives the plans of the host model above on GB300."""
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("plans are recorded for 152 SMs")
    shp = W.WORKLOADS[name]
    lens = W.draw_seq_lens(shp, np.random.default_rng(shp.seed))
    p = params(shp.batch, shp.q_len, shp.num_q_heads, shp.num_kv_heads, int(lens.max()),
               shp.page_size if shp.paged else 0, shp.causal)
    if getattr(shp, "kv_fp8", False):
        p.flags |= binding.DA_FLAG_KV_FP8_E4M3
    assert binding.decode_attn_plan(p, lens) == BENCH_PLANS[name]


@pytest.mark.parametrize("batch,hkv,want", [(1, 8, 16), (1, 32, 16), (1, 64, 9), (2, 64, 4),
                                            (4, 64, 2), (19, 32, 1), (64, 32, 1)])
def test_equal_lengths_fill_one_wave_of_at_most_16_chunks(batch, hkv, want):
    L = 65536
    p = params(batch, 1, hkv, hkv, L, 0)
    lens = np.full(batch, L, np.int32)
    S, chunk = binding.decode_attn_plan_slots(p, lens, NARROW_SLOTS)
    assert S == want == min(16, max(1, NARROW_SLOTS // (batch * hkv)))
    assert chunk % 16 == 0 and S * chunk >= L > (S - 1) * chunk
    # without host lengths the planner assumes max_seq_len everywhere
    assert binding.decode_attn_plan_slots(p, None, NARROW_SLOTS) == (S, chunk)


@pytest.mark.parametrize("q_len,hq,hkv", [(1, 32, 8), (4, 32, 8), (1, 64, 8), (8, 64, 8),
                                          (16, 64, 8)])
def test_ragged_chunks_hold_the_per_row_floor_when_the_gpu_is_full(q_len, hq, hkv):
    rng = np.random.default_rng(7)
    lens = rng.integers(1024, 16385, size=256).astype(np.int32)
    r = rows(hq, hkv, q_len)
    p = params(256, q_len, hq, hkv, int(lens.max()), 16, causal=q_len > 1)
    S, chunk = binding.decode_attn_plan_slots(p, lens, slots_for(r))
    floor = max(256, (256 if r > 16 else 64) * r)
    msl = int(lens.max())
    # chunks of at least `floor` tokens: no more splits than that allows (the
    # final chunk is max_seq_len / splits rounded up to 16 tokens)
    assert S <= -(-msl // floor)
    assert chunk % 16 == 0 and S * chunk >= msl > (S - 1) * chunk
    assert chunks(lens, chunk, hkv) >= slots_for(r)


def test_ragged_chunks_aim_at_about_eight_waves():
    rng = np.random.default_rng(8)
    lens = rng.integers(512, 32769, size=64).astype(np.int32)
    p = params(64, 1, 32, 8, int(lens.max()), 16)
    S, chunk = binding.decode_attn_plan_slots(p, lens, NARROW_SLOTS)
    waves = chunks(lens, chunk, 8) / NARROW_SLOTS
    assert 6 <= waves <= 10, waves


@pytest.mark.parametrize("lens,q_len", [([11700, 15700], 8), ([9000, 16000, 12000, 14000], 16)])
def test_small_ragged_batch_still_fills_every_slot(lens, q_len):
    # a few requests with 64-128 query rows per kv head: the tokens-per-row
    # floor (8192 or 16384) would leave 16-40 chunks for 152 SMs, so the
    # chunk shrinks until the batch has a chunk for every resident CTA
    lens = np.array(lens, np.int32)
    p = params(len(lens), q_len, 64, 8, int(lens.max()), 16, causal=True)
    S, chunk = binding.decode_attn_plan_slots(p, lens, WIDE_SLOTS)
    assert 256 <= chunk < 8192
    assert chunks(lens, chunk, 8) >= WIDE_SLOTS


@pytest.mark.parametrize("max_seq_len,want", [(0, 1), (16, 1), (255, 1), (511, 1), (512, 2)])
def test_short_contexts_keep_chunks_of_at_least_256_tokens(max_seq_len, want):
    p = params(1, 1, 8, 8, max_seq_len, 0)
    S, chunk = binding.decode_attn_plan_slots(p, None, NARROW_SLOTS)
    assert S == want
    assert chunk % 16 == 0 and chunk >= 16


def test_plan_arguments_are_checked():
    p = params(1, 1, 8, 8, 4096, 0)
    for bad_slots in (0, -5, 2**31 + 1, 2**62):
        with pytest.raises(binding.DecodeAttnError):
            binding.decode_attn_plan_slots(p, None, bad_slots)
    # the largest accepted count plans without overflow (equal and ragged lengths)
    assert binding.decode_attn_plan_slots(p, None, 2**31)[0] >= 1
    lens = np.array([100, 4096], np.int32)
    p2 = params(2, 1, 8, 8, 4096, 16)
    assert binding.decode_attn_plan_slots(p2, lens, 2**31)[0] >= 1
    bad = params(1, 1, 8, 8, 4096, 0)
    bad.head_dim = 64
    with pytest.raises(binding.DecodeAttnError):
        binding.decode_attn_plan_slots(bad, None, NARROW_SLOTS)


def brute_force_plan(lens, hkv, rows, msl, slots):
    """The planner's rule as its documentation states it, with the split
    search done by brute force: every candidate chunk length tested."""
    lens = np.asarray(lens, np.int64)
    L = np.clip(lens, 0, msl)
    uniform = bool(np.all(lens == lens[0]))
    pairs = max(len(lens), 1) * hkv
    max_tiles = -(-max(msl, 1) // 16)
    if uniform:
        splits = min(slots // pairs, 16) if pairs < slots else 1
    else:
        per_cta = -(-int(L.sum()) * hkv // (8 * slots))
        min_chunk = max((256 if rows > 16 else 64) * rows, 256)
        hi = max(per_cta, min_chunk)
        cs = np.arange(hi, 256, -1, dtype=np.int64)          # (256, hi], longest first
        counts = np.where(L[:, None] > 0, -(-L[:, None] // cs[None, :]), 1).sum(axis=0) * hkv
        ok = np.nonzero(counts >= slots)[0]
        target = int(cs[ok[0]]) if len(ok) else 256
        splits = -(-max(msl, 1) // target)
    splits = max(1, min(splits, max(msl // 256, 1), max_tiles))
    chunk = -(-(-(-max(msl, 1) // splits)) // 16) * 16
    return max(1, -(-msl // chunk)), chunk              # (chunks at max_seq_len, length)


@pytest.mark.parametrize("seed", range(40))
def test_split_search_equals_brute_force(seed):
    """The host planner's split search (test the top, then bisect) gives the
    length a scan of every candidate gives, over ragged and equal batches,
    narrow and wide query groups and slot counts that make it search."""
    rng = np.random.default_rng(300 + seed)
    B = int(rng.integers(1, 65))
    hkv = int(rng.choice([1, 2, 8]))
    q_len, hq = [(1, 4 * hkv), (4, 4 * hkv), (8, 8 * hkv), (16, 8 * hkv)][int(rng.integers(0, 4))]
    hi = int(rng.choice([300, 3000, 20000, 50000]))
    lens = rng.integers(0, hi, B).astype(np.int32)
    if rng.random() < 0.2:
        lens[:] = lens[0]                                  # equal lengths
    msl = max(16, int(lens.max()))
    rows = hq // hkv * q_len
    slots = int(rng.choice([152, 608, 1000, 5000]))
    p = params(B, q_len, hq, hkv, msl, 16, causal=False)
    got = binding.decode_attn_plan_slots(p, lens, slots)
    assert got == brute_force_plan(lens, hkv, rows, msl, slots), (B, hkv, rows, msl, slots)
