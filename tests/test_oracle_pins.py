"""Pins of the fp64 oracle to facts it does not compute itself.

Each test checks the oracle against something the pages or mathematics fix:
the worked example printed on the pages, closed forms, invariants, library
routines (scipy) on tiny inputs, and the pages' own error bound for the tiled
recurrence.  Together they are chosen so that a plausible slip in the oracle
(a wrong GQA head map, a page/slot index swap, a dropped causal offset, a
missing scale, a sign error in a merge weight) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
from split_kv_decode_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals[k] = [float(x) for x in v.split()]
    return vals


def bf16(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def f32(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def one_head_problem(scores_basis, values, D=128):
    """Single request, single head, contiguous cache whose scores (scale 1)
    are exactly `scores_basis`: q = e_0 and k_j = s_j * e_0."""
    L = len(scores_basis)
    q = np.zeros((1, 1, 1, D), np.float32)
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, L, 1, D), np.float32)
    k[0, :, 0, 0] = scores_basis
    v = np.asarray(values, np.float32).reshape(1, L, 1, D)
    return bf16(q), bf16(k), bf16(v), np.array([L], np.int32)


# ---------------------------------------------------------------------------
# 1. The pages' worked example of the two-block merge
# ---------------------------------------------------------------------------
def test_worked_example_merge_matches_printed_values():
    g = read_golden("online_softmax_worked_example.txt")
    # merge of the printed block statistics (lse_s = m_s + ln l_s)
    lse_a = g["m_a"][0] + math.log(g["l_a"][0])
    lse_b = g["m_b"][0] + math.log(g["l_b"][0])
    o_a = np.zeros((1, 2, 4))
    out, lse = oracle.merge_partials(o_a, np.array([[lse_a, lse_b]]))
    l_new = math.exp(lse[0] - g["m_new"][0])
    assert abs(l_new - g["l_new"][0]) <= 1e-4
    assert abs(math.exp(g["m_a"][0] - g["m_new"][0]) - g["decay_a"][0]) <= 1e-4


def test_worked_example_oracle_statistics_of_each_block_and_whole_row():
    g = read_golden("online_softmax_worked_example.txt")
    row = g["row_a"] + g["row_b"]
    D = 128
    vals = np.random.default_rng(0).standard_normal((4, D))
    q, k, v, L = one_head_problem(row, vals)
    common = dict(num_kv_heads=1, scale=1.0)
    _, lse_full = oracle.decode_attention(q, k, v, L, **common)
    _, lse_a = oracle.decode_attention(q, k, v, L, key_lo=0, key_hi=2, **common)
    _, lse_b = oracle.decode_attention(q, k, v, L, key_lo=2, key_hi=4, **common)
    # block statistics as printed: l_s = exp(lse_s - m_s)
    assert abs(math.exp(lse_a.item() - g["m_a"][0]) - g["l_a"][0]) <= 1e-4
    assert abs(math.exp(lse_b.item() - g["m_b"][0]) - g["l_b"][0]) <= 1e-4
    assert abs(math.exp(lse_full.item() - g["m_new"][0]) - g["l_truth"][0]) <= 1e-4
    # and the exact closed form e^-3 + e^-1 + e^-2 + 1
    exact = math.exp(-3) + math.exp(-1) + math.exp(-2) + 1.0
    assert abs(math.exp(lse_full.item() - 5.0) - exact) <= 1e-14


# ---------------------------------------------------------------------------
# 2. Closed forms and special cases
# ---------------------------------------------------------------------------
def test_single_key_returns_its_value_exactly():
    rng = np.random.default_rng(1)
    D = 128
    q = bf16(rng.standard_normal((2, 1, 4, D)))
    k = bf16(rng.standard_normal((2, 5, 2, D)))
    v = bf16(rng.standard_normal((2, 5, 2, D)))
    L = np.array([1, 1], np.int32)
    out, lse = oracle.decode_attention(q, k, v, L, num_kv_heads=2)
    for b in range(2):
        for h in range(4):
            kvh = h // 2
            np.testing.assert_array_equal(out[b, 0, h], f32(v[b, 0, kvh]))
            s0 = np.dot(f32(q[b, 0, h]), f32(k[b, 0, kvh])) / math.sqrt(D)
            assert abs(lse[b, 0, h] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    D, L = 128, 37
    q = bf16(rng.standard_normal((1, 1, 1, D)))
    key = rng.standard_normal(D)
    k = bf16(np.broadcast_to(key, (1, L, 1, D)))
    v = bf16(rng.standard_normal((1, L, 1, D)))
    out, lse = oracle.decode_attention(q, k, v, np.array([L], np.int32),
                                       num_kv_heads=1)
    np.testing.assert_allclose(out[0, 0, 0], f32(v)[0, :, 0].mean(0), rtol=0,
                               atol=1e-14)
    s = np.dot(f32(q[0, 0, 0]), f32(k[0, 0, 0])) / math.sqrt(D)
    assert abs(lse.item() - (s + math.log(L))) <= 1e-12


def test_zero_query_gives_mean_and_log_length():
    rng = np.random.default_rng(3)
    D, L = 128, 50
    q = bf16(np.zeros((1, 1, 2, D)))
    k = bf16(rng.standard_normal((1, L, 1, D)) * 5)
    v = bf16(rng.standard_normal((1, L, 1, D)))
    out, lse = oracle.decode_attention(q, k, v, np.array([L], np.int32),
                                       num_kv_heads=1)
    for h in range(2):
        np.testing.assert_allclose(out[0, 0, h], f32(v)[0, :, 0].mean(0),
                                   atol=1e-14, rtol=0)
        assert abs(lse[0, 0, h] - math.log(L)) <= 1e-14


@pytest.mark.parametrize("scale", [1.0, 0.5, 1 / math.sqrt(128)])
def test_two_keys_logistic_weights_and_scale(scale):
    # scores (before scale) a and b: weight of key 1 = 1 / (1 + e^{scale(a-b)})
    a, b = 3.0, -1.5
    D = 128
    vals = np.zeros((2, D))
    vals[0, :] = 1.0
    vals[1, :] = -2.0
    q, k, v, L = one_head_problem([a, b], vals)
    out, lse = oracle.decode_attention(q, k, v, L, num_kv_heads=1, scale=scale)
    w1 = 1.0 / (1.0 + math.exp(scale * (a - b)))
    assert abs(out[0, 0, 0, 0] - ((1 - w1) * 1.0 + w1 * -2.0)) <= 1e-15
    expect_lse = math.log(math.exp(scale * a) + math.exp(scale * b))
    assert abs(lse.item() - expect_lse) <= 1e-15


def test_empty_row_is_zero_with_minus_inf_lse():
    rng = np.random.default_rng(4)
    D = 128
    q = bf16(rng.standard_normal((2, 1, 2, D)))
    k = bf16(rng.standard_normal((2, 8, 1, D)))
    out, lse = oracle.decode_attention(q, k, k, np.array([0, 3], np.int32),
                                       num_kv_heads=1)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# ---------------------------------------------------------------------------
# 3. Brute force against scipy's softmax / logsumexp on tiny inputs
# ---------------------------------------------------------------------------
def logical_kv(inp, b, kvh):
    """Logical key/value rows of request b (test-side gather, numpy)."""
    L = int(inp.seq_lens[b])
    if inp.block_table is None:
        return f32(inp.k_cache[b, :L, kvh]), f32(inp.v_cache[b, :L, kvh])
    j = np.arange(L)
    pages = inp.block_table[b, j // inp.page_size]
    slots = j % inp.page_size
    return f32(inp.k_cache[pages, slots, kvh]), f32(inp.v_cache[pages, slots, kvh])


@pytest.mark.parametrize("G,q_len,causal,paged", [
    (1, 1, False, True), (4, 1, False, True), (8, 1, False, False),
    (4, 4, True, True), (2, 3, True, False), (4, 4, False, True)])
def test_brute_force_tiny_against_scipy(G, q_len, causal, paged):
    shp = W.small_shape(batch=3, q_len=q_len, num_q_heads=2 * G, num_kv_heads=2,
                        lo=4, hi=40, paged=paged, causal=causal, seed=11 + G)
    inp = W.make_host_inputs(shp)
    out, lse = oracle.decode_attention_inputs(inp)
    D = shp.head_dim
    for b in range(shp.batch):
        L = int(inp.seq_lens[b])
        for t in range(q_len):
            for h in range(shp.num_q_heads):
                kvh = h // G
                K, V = logical_kv(inp, b, kvh)
                n = L - q_len + 1 + t if causal else L
                s = K[:n] @ f32(inp.q[b, t, h]) * shp.scale
                np.testing.assert_allclose(out[b, t, h], softmax(s) @ V[:n],
                                           rtol=0, atol=1e-13)
                assert abs(lse[b, t, h] - logsumexp(s)) <= 1e-12
    assert out.shape == (shp.batch, q_len, shp.num_q_heads, D)


# ---------------------------------------------------------------------------
# 4. Invariants: paging, GQA map, causal offsets, permutation, V scaling
# ---------------------------------------------------------------------------
def test_shuffled_pages_equal_contiguous_layout_bit_exact():
    shp = W.small_shape(batch=4, num_q_heads=8, num_kv_heads=2, lo=1, hi=200,
                        paged=True, page_size=16, seed=21)
    shuffled = W.make_host_inputs(shp, shuffle=True)
    # rebuild the same logical sequences as a contiguous [B, Lmax, Hkv, D] cache
    Lmax = int(shuffled.seq_lens.max())
    kc = np.zeros((shp.batch, Lmax, 2, 128), np.uint16)
    vc = np.zeros_like(kc)
    for b in range(shp.batch):
        L = int(shuffled.seq_lens[b])
        for j in range(L):
            p = shuffled.block_table[b, j // 16]
            kc[b, j] = shuffled.k_cache[p, j % 16]
            vc[b, j] = shuffled.v_cache[p, j % 16]
    o1, l1 = oracle.decode_attention_inputs(shuffled)
    o2, l2 = oracle.decode_attention(shuffled.q, kc, vc, shuffled.seq_lens,
                                     num_kv_heads=2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def paginate(kc, vc, seq_lens, page_size, rng):
    """Scatter contiguous [B, Lmax, Hkv, D] caches into shuffled pages."""
    B, _, Hkv, D = kc.shape
    need = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    P = sum(need)
    perm = rng.permutation(P)
    kp = np.zeros((P, page_size, Hkv, D), kc.dtype)
    vp = np.zeros_like(kp)
    bt = np.full((B, max(need)), -1, np.int32)
    off = 0
    for b in range(B):
        for i in range(need[b]):
            p = perm[off + i]
            bt[b, i] = p
            seg = slice(i * page_size, min((i + 1) * page_size, int(seq_lens[b])))
            n = seg.stop - seg.start
            kp[p, :n] = kc[b, seg]
            vp[p, :n] = vc[b, seg]
        off += need[b]
    return kp, vp, bt


@pytest.mark.parametrize("page_size", [16, 32, 64])
def test_paged_layouts_of_any_page_size_equal_contiguous(page_size):
    rng = np.random.default_rng(5)
    B, Lmax, Hkv, D = 3, 150, 2, 128
    kc = bf16(rng.standard_normal((B, Lmax, Hkv, D)))
    vc = bf16(rng.standard_normal((B, Lmax, Hkv, D)))
    q = bf16(rng.standard_normal((B, 1, 4, D)))
    lens = np.array([150, 1, 77], np.int32)
    kp, vp, bt = paginate(kc, vc, lens, page_size, rng)
    o1, l1 = oracle.decode_attention(q, kc, vc, lens, num_kv_heads=Hkv)
    o2, l2 = oracle.decode_attention(q, kp, vp, lens, num_kv_heads=Hkv,
                                     block_table=bt, page_size=page_size)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_gqa_maps_contiguous_head_groups():
    # V of kv head i is the constant i + 1, so out of query head h is h//G + 1
    D, Hkv, G, L = 128, 4, 3, 9
    rng = np.random.default_rng(6)
    q = bf16(rng.standard_normal((1, 1, Hkv * G, D)))
    k = bf16(rng.standard_normal((1, L, Hkv, D)))
    vv = np.zeros((1, L, Hkv, D), np.float32)
    for i in range(Hkv):
        vv[:, :, i, :] = i + 1
    out, _ = oracle.decode_attention(q, k, bf16(vv), np.array([L], np.int32),
                                     num_kv_heads=Hkv)
    for h in range(Hkv * G):
        np.testing.assert_allclose(out[0, 0, h], h // G + 1, rtol=0, atol=1e-14)


def test_causal_token_t_equals_plain_decode_at_shorter_length():
    shp = W.small_shape(batch=2, q_len=4, num_q_heads=8, num_kv_heads=2,
                        lo=20, hi=90, paged=True, causal=True, seed=8)
    inp = W.make_host_inputs(shp)
    out, lse = oracle.decode_attention_inputs(inp)
    for t in range(4):
        q1 = np.ascontiguousarray(inp.q[:, t:t + 1])
        lens = inp.seq_lens - 3 + t
        o1, l1 = oracle.decode_attention(
            q1, inp.k_cache, inp.v_cache, lens, num_kv_heads=2,
            block_table=inp.block_table, page_size=16)
        np.testing.assert_array_equal(out[:, t], o1[:, 0])
        np.testing.assert_array_equal(lse[:, t], l1[:, 0])
    # the last token sees all L keys: identical to the non-causal result
    nc, lnc = oracle.decode_attention(
        inp.q, inp.k_cache, inp.v_cache, inp.seq_lens, num_kv_heads=2,
        block_table=inp.block_table, page_size=16, causal=False)
    np.testing.assert_array_equal(out[:, 3], nc[:, 3])
    assert not np.array_equal(out[:, 0], nc[:, 0])


def test_permuting_key_value_pairs_leaves_result_unchanged():
    rng = np.random.default_rng(9)
    D, L = 128, 64
    q = bf16(rng.standard_normal((1, 1, 2, D)))
    k = bf16(rng.standard_normal((1, L, 1, D)))
    v = bf16(rng.standard_normal((1, L, 1, D)))
    perm = rng.permutation(L)
    o1, l1 = oracle.decode_attention(q, k, v, np.array([L], np.int32), num_kv_heads=1)
    o2, l2 = oracle.decode_attention(q, np.ascontiguousarray(k[:, perm]),
                                     np.ascontiguousarray(v[:, perm]),
                                     np.array([L], np.int32), num_kv_heads=1)
    np.testing.assert_allclose(o1, o2, atol=1e-14, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-13, rtol=0)
    # but permuting values alone changes it
    o3, _ = oracle.decode_attention(q, k, np.ascontiguousarray(v[:, perm]),
                                    np.array([L], np.int32), num_kv_heads=1)
    assert np.abs(o3 - o1).max() > 1e-3


def test_output_is_linear_in_values():
    shp = W.small_shape(batch=2, lo=5, hi=60, seed=10)
    inp = W.make_host_inputs(shp)
    o1, l1 = oracle.decode_attention_inputs(inp)
    v2 = bf16(f32(inp.v_cache) * 2.0)   # exact in bf16
    o2, l2 = oracle.decode_attention(inp.q, inp.k_cache, v2, inp.seq_lens,
                                     num_kv_heads=2, block_table=inp.block_table,
                                     page_size=16)
    np.testing.assert_array_equal(o2, 2.0 * o1)
    np.testing.assert_array_equal(l1, l2)


def test_out_of_range_page_is_reported():
    shp = W.small_shape(batch=2, lo=20, hi=40, seed=12)
    inp = W.make_host_inputs(shp)
    bt = inp.block_table.copy()
    bt[1, 0] = inp.num_pages   # one past the end
    with pytest.raises(ValueError, match="code -2"):
        oracle.decode_attention(inp.q, inp.k_cache, inp.v_cache, inp.seq_lens,
                                num_kv_heads=2, block_table=bt, page_size=16)


# ---------------------------------------------------------------------------
# 5. Chunked merge == one shot (the pages' proof), and the pages' error bound
# ---------------------------------------------------------------------------
def test_merge_of_key_chunks_equals_one_shot():
    shp = W.small_shape(batch=3, q_len=2, num_q_heads=8, num_kv_heads=2,
                        lo=50, hi=300, causal=True, seed=13)
    inp = W.make_host_inputs(shp)
    full_o, full_l = oracle.decode_attention_inputs(inp)
    rng = np.random.default_rng(14)
    cuts = sorted(rng.choice(np.arange(1, 300), size=4, replace=False).tolist())
    bounds = [0] + cuts + [10**9]
    parts = [oracle.decode_attention_inputs(inp, key_lo=a, key_hi=b)
             for a, b in zip(bounds[:-1], bounds[1:])]
    po = np.stack([p[0] for p in parts], axis=-2)
    pl = np.stack([p[1] for p in parts], axis=-1)
    mo, ml = oracle.merge_partials(po, pl)
    np.testing.assert_allclose(mo, full_o, atol=1e-13, rtol=0)
    np.testing.assert_allclose(ml, full_l, atol=1e-12, rtol=0)


def test_merge_ignores_empty_chunks_and_all_empty_row():
    po = np.random.default_rng(15).standard_normal((2, 3, 128))
    pl = np.array([[-np.inf, 1.0, -np.inf], [-np.inf, -np.inf, -np.inf]])
    out, lse = oracle.merge_partials(po, pl)
    np.testing.assert_array_equal(out[0], po[0, 1])
    assert lse[0] == 1.0
    assert np.all(out[1] == 0) and np.isneginf(lse[1])


def test_merge_nvalid_uses_leading_splits_only():
    rng = np.random.default_rng(16)
    po = rng.standard_normal((2, 4, 128))
    pl = rng.standard_normal((2, 4))
    out, lse = oracle.merge_partials(po, pl, nvalid=np.array([2, 4]))
    o2, l2 = oracle.merge_partials(po[:1, :2], pl[:1, :2])
    np.testing.assert_array_equal(out[0], o2[0])
    assert lse[0] == l2[0]


def test_tiled_online_recurrence_within_pages_error_bound():
    """The pages check their tiled forward against standard attention to a max
    error below 1e-10 in fp64 (N=256 rows, d=64, 64-wide blocks).  Here the
    running-max / running-sum recurrence of §1.2 is stepped over 64-key blocks
    for each of 256 query rows and compared to the oracle."""
    rng = np.random.default_rng(42)
    N, D = 256, 64
    Q = f32(bf16(rng.standard_normal((N, D))))
    K = f32(bf16(rng.standard_normal((N, D))))
    V = f32(bf16(rng.standard_normal((N, D))))
    scale = 1.0 / math.sqrt(D)
    # oracle: each query row as one decode request over the same N keys
    q = bf16(Q).reshape(N, 1, 1, D)
    kc = np.broadcast_to(bf16(K).reshape(1, N, 1, D), (N, N, 1, D)).copy()
    vc = np.broadcast_to(bf16(V).reshape(1, N, 1, D), (N, N, 1, D)).copy()
    ref, _ = oracle.decode_attention(q, kc, vc, np.full(N, N, np.int32),
                                     num_kv_heads=1, scale=scale)
    ref = ref.reshape(N, D)
    # running statistics over 64-key blocks, division deferred to the end
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    acc = np.zeros((N, D))
    for j0 in range(0, N, 64):
        S = (Q @ K[j0:j0 + 64].T) * scale
        m_new = np.maximum(m, S.max(axis=1))
        P = np.exp(S - m_new[:, None])
        alpha = np.exp(m - m_new)
        acc = acc * alpha[:, None] + P @ V[j0:j0 + 64]
        l = l * alpha + P.sum(axis=1)
        m = m_new
    tiled = acc / l[:, None]
    assert np.abs(tiled - ref).max() < 1e-10


# ---------------------------------------------------------------- FP8 E4M3 caches
def test_e4m3_decoding_matches_torch_float8_for_every_code():
    """The oracle's E4M3 decoder (written from the format definition) against
    PyTorch's float8_e4m3fn for all 256 codes; NaN exactly at S.1111.111."""
    torch = pytest.importorskip("torch")
    mine = oracle.e4m3_values()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))   # -0 is 0x80


def test_e4m3_closed_forms():
    v = oracle.e4m3_values()
    assert v[0x38] == 1.0 and v[0xB8] == -1.0          # exponent field 7 = bias
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0      # largest finite value
    assert v[0x08] == 2.0 ** -6                        # smallest normal
    assert v[0x01] == 2.0 ** -9                        # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9                    # largest subnormal
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x00] == 0.0 and np.signbit(v[0x80])


def _fp8_problem(seed, k_scale, v_scale, paged=True, causal=True):
    shp = W.small_shape("f8pin", batch=3, q_len=2, num_q_heads=8, num_kv_heads=2,
                        lo=3, hi=70, paged=paged, causal=causal, seed=seed, kv_fp8=True)
    inp = W.make_host_inputs(shp)
    inp.k_scale, inp.v_scale = k_scale, v_scale
    return inp


@pytest.mark.parametrize("paged", [True, False])
def test_fp8_cache_equals_bf16_cache_of_the_decoded_values(paged):
    """With power-of-two scales every k_scale * E4M3 value is a bf16 value, so
    the FP8 path must give exactly the bf16 path on those values."""
    inp = _fp8_problem(50, 2.0 ** -3, 2.0 ** 2, paged=paged)
    vals = oracle.e4m3_values()
    kb = bf16(vals[inp.k_cache] * inp.k_scale)
    vb = bf16(vals[inp.v_cache] * inp.v_scale)
    assert np.array_equal(f32(kb).astype(np.float64), vals[inp.k_cache] * inp.k_scale)
    o8, l8 = oracle.decode_attention_inputs(inp)
    s = inp.shape
    o16, l16 = oracle.decode_attention(
        inp.q, kb, vb, inp.seq_lens, num_kv_heads=s.num_kv_heads,
        block_table=inp.block_table, page_size=inp.page_size, num_pages=inp.num_pages,
        scale=s.scale, causal=s.causal)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)


def test_fp8_value_scale_is_linear_and_key_scale_scales_the_scores():
    inp = _fp8_problem(51, 0.01, 0.02)
    o1, l1 = oracle.decode_attention_inputs(inp)
    inp.v_scale = 0.04                       # doubling v_scale doubles the output
    o2, l2 = oracle.decode_attention_inputs(inp)
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-14, atol=1e-300)
    assert np.array_equal(l1, l2)
    # k_scale enters only as a factor on the scores: k_scale * c with softmax
    # scale s equals k_scale c' = k_scale * c / 2 with softmax scale 2 s
    s = inp.shape
    o3, l3 = oracle.decode_attention(
        inp.q, inp.k_cache, inp.v_cache, inp.seq_lens, num_kv_heads=s.num_kv_heads,
        block_table=inp.block_table, page_size=inp.page_size, num_pages=inp.num_pages,
        scale=2 * s.scale, causal=s.causal, kv_fp8=True, k_scale=0.005, v_scale=0.04)
    np.testing.assert_allclose(o3, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l3, l2, rtol=1e-12, atol=1e-14)


def test_fp8_workload_recipe_quantises_within_half_an_e4m3_step():
    """Input-recipe check: every stored byte decodes to within half an E4M3
    step of x / scale (round to nearest), and the largest |x| maps to 448."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    b, sc = W.quantize_e4m3(x)
    vals = oracle.e4m3_values()[b]
    y = x.astype(np.float64) / sc
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))) - 3)
    assert np.all(np.abs(vals - y) <= ulp / 2 + 1e-12)
    assert np.abs(vals).max() == 448.0
