"""GPU check: cache contents a call must not use -- rows past each request's
length, the unused slots of its last page, pages no request references -- may
hold anything, NaN included.  The kernels mask the scores of such keys and
zero their value rows before the P.V product (NaN * 0 is NaN), so every
kernel variant must return the same bits with those rows poisoned as with
them clean.  All calls go through the C ABI."""
import numpy as np
import pytest

from split_kv_decode_attention_gb300 import workloads as W

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


# (id, batch, q_len, Hq, Hkv, paged, causal, fp8, num_splits, two_pass)
# rows per KV head = q_len * Hq / Hkv: 4 and 16 run the warp-MMA kernel, 64
# and 128 the tcgen05 kernel; num_splits 0 plans on the device (listed
# variants); fixed split counts with two_pass keep the partials + combine
# form, without it small calls take the cluster merge
CASES = [
    ("rows4_contiguous", 3, 1, 8, 2, False, False, False, 3, False),
    ("rows4_paged_two_pass", 3, 1, 8, 2, True, False, False, 4, True),
    ("rows4_paged_device_plan", 3, 1, 8, 2, True, False, False, 0, False),
    ("rows16_paged_causal", 3, 4, 16, 4, True, True, False, 4, True),
    ("rows4_fp8_paged", 3, 1, 8, 2, True, False, True, 3, True),
    ("rows16_fp8_contiguous", 3, 4, 16, 4, False, True, True, 2, False),
    ("rows64_paged_causal", 3, 8, 64, 8, True, True, False, 2, True),
    ("rows64_fp8_paged", 3, 8, 64, 8, True, True, True, 2, True),
    ("rows64_device_plan", 3, 8, 64, 8, True, True, False, 0, False),
    ("rows128_contiguous", 2, 16, 64, 8, False, True, False, 3, True),
]


def _poison(inp, shape):
    """Copies of the caches whose unused rows hold NaN (bf16 0x7FC0, E4M3 0x7F)."""
    lens = inp.seq_lens.cpu().numpy()
    k = inp.k_cache.clone()
    v = inp.v_cache.clone()
    nan_k = k.view(torch.uint8) if shape.kv_fp8 else k.view(torch.int16)
    nan_v = v.view(torch.uint8) if shape.kv_fp8 else v.view(torch.int16)
    bits = 0x7F if shape.kv_fp8 else 0x7FC0
    if shape.paged:
        ps = inp.page_size
        used = torch.zeros(k.shape[:2], dtype=torch.bool)
        bt = inp.block_table.cpu().numpy()
        for b, L in enumerate(lens):
            for i in range(-(-int(L) // ps)):
                used[int(bt[b, i]), :min(ps, int(L) - i * ps)] = True
        unused = (~used).to(k.device)
        nan_k[unused] = bits
        nan_v[unused] = bits
    else:
        for b, L in enumerate(lens):
            nan_k[b, int(L):] = bits
            nan_v[b, int(L):] = bits
    return k, v


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_unused_cache_rows_never_reach_the_output(binding, case):
    _, B, T, Hq, Hkv, paged, causal, fp8, splits, two_pass = case
    # lengths down to q_len and up to a few tiles past a 64-key stage, so
    # partial tiles, partial stages and partial pages all occur
    shape = W.small_shape("poison", batch=B, q_len=T, num_q_heads=Hq, num_kv_heads=Hkv,
                          lo=T, hi=300, paged=paged, causal=causal, seed=91 + B * T,
                          kv_fp8=fp8)
    inp = W.make_device_inputs(shape)
    # some request ends inside a 16-token tile, so whole-tile copies bring
    # poisoned rows on chip
    assert any(int(L) % 16 for L in inp.seq_lens.cpu().numpy())
    kw = dict(max_seq_len=inp.max_seq_len, causal=causal, num_splits=splits,
              two_pass=two_pass, k_scale=inp.k_scale, v_scale=inp.v_scale)
    o1, l1 = binding.decode_attn(inp.q, inp.k_cache, inp.v_cache, inp.block_table,
                                 inp.seq_lens, **kw)
    kp, vp = _poison(inp, shape)
    assert not torch.equal(kp.view(torch.uint8), inp.k_cache.view(torch.uint8))
    o2, l2 = binding.decode_attn(inp.q, kp, vp, inp.block_table, inp.seq_lens, **kw)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o2.float()).all())
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
