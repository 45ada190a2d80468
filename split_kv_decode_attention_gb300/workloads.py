"""Seeded synthetic decode-attention workloads.

This module only *generates inputs*: query rows, bf16 K/V caches (contiguous or
paged), ragged sequence lengths and shuffled block tables.  It holds none of
the attention arithmetic, so that the fp64 oracle and the CUDA path can both
consume the same inputs without sharing any code that computes a result.

Shapes follow the decode problem statement of the pages:
  * one query token (or a few speculative tokens) per request attends over a
    long KV history ("Capstone FlashAttention", §2.3 FlashDecoding; the
    inference-engine chapter "12. attention kernels", decode-attention section);
  * GQA: 32 query heads in 8 groups share 8 KV heads ("Capstone
    FlashAttention", §4.2);
  * PagedAttention: fixed 16-token physical blocks, a per-request block table,
    physically scattered but logically contiguous ("Capstone FlashAttention",
    §4.1 and hands-on lab 2).

Numbers are drawn from numpy's PCG64 (host) or torch's CUDA generator (device,
used for the multi-GB workloads); both round fp32 -> bf16 with
round-to-nearest-even.  Values are stored as raw bf16 bit patterns (uint16) on
the host so that no library's bf16 type is involved in the oracle's reading of
them.

FP8 caches (`kv_fp8` recipes): the same normal K / V values, quantised per
cache to OCP FP8 E4M3 with one fp32 scale, scale = max|x| / 448 (the largest
E4M3 value), bytes = E4M3(x / scale) rounded to nearest even by torch's
float8_e4m3fn conversion -- the cache format with explicit scaling factors
("Capstone FlashAttention", §2.2 FP8 with scaling; the CUTLASS split-KV post,
§5.8).  Bytes are stored as uint8.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

HEAD_DIM = 128
PAGE_TILE = 16  # tokens per physical page in every paged workload below


# ---------------------------------------------------------------------------
# bf16 bit conversions (input preparation only)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return the
    16-bit patterns as uint16.  NaN stays NaN (quiet)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> 16) & 1
    rounded = ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)
    if nan.any():
        rounded = np.where(nan, ((u >> 16) | 0x40).astype(np.uint16), rounded)
    return rounded


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Workload description
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class DecodeShape:
    """One synthetic decode-attention workload recipe."""

    name: str
    batch: int
    q_len: int
    num_q_heads: int
    num_kv_heads: int
    seq_len_lo: int          # seq_lens ~ integers uniform on [lo, hi] (inclusive)
    seq_len_hi: int
    paged: bool              # False: contiguous [B, max_seq_len, Hkv, D] cache
    page_size: int = PAGE_TILE
    causal: bool = False     # mask among the q_len new tokens
    peaked_key_fraction: float = 0.0   # fraction of K rows multiplied by 8
    head_dim: int = HEAD_DIM
    seed: int = 0
    kv_fp8: bool = False     # caches in FP8 E4M3 with one scale each

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return float(1.0 / np.sqrt(self.head_dim))


# The five workloads (sizes, head counts, length mixes and value
# distributions), seeds 1000 + index.
WORKLOADS = {
    "c1_b1_h32kv8_L4096": DecodeShape(
        "c1_b1_h32kv8_L4096", batch=1, q_len=1, num_q_heads=32, num_kv_heads=8,
        seq_len_lo=4096, seq_len_hi=4096, paged=False, seed=1001),
    "c2_b1_mha32_L131072": DecodeShape(
        "c2_b1_mha32_L131072", batch=1, q_len=1, num_q_heads=32, num_kv_heads=32,
        seq_len_lo=131072, seq_len_hi=131072, paged=False, seed=1002),
    "c3_b64_h32kv8_L512-32768_paged": DecodeShape(
        "c3_b64_h32kv8_L512-32768_paged", batch=64, q_len=1, num_q_heads=32,
        num_kv_heads=8, seq_len_lo=512, seq_len_hi=32768, paged=True, seed=1003),
    "c4_b256_h64kv8_L128-4096_paged_peaked": DecodeShape(
        "c4_b256_h64kv8_L128-4096_paged_peaked", batch=256, q_len=1,
        num_q_heads=64, num_kv_heads=8, seq_len_lo=128, seq_len_hi=4096,
        paged=True, peaked_key_fraction=0.01, seed=1004),
    "c5_b32_q4_causal_h32kv8_L1024-16384_paged": DecodeShape(
        "c5_b32_q4_causal_h32kv8_L1024-16384_paged", batch=32, q_len=4,
        num_q_heads=32, num_kv_heads=8, seq_len_lo=1024, seq_len_hi=16384,
        paged=True, causal=True, seed=1005),
}
WORKLOAD_ORDER = list(WORKLOADS)

# Wider speculative verify (G x q_len = 64 and 128 query rows per KV head):
# the same synthetic recipe as c5, with 8 and 16 draft tokens.
WIDE_WORKLOADS = {
    "w64_b32_q8_h64kv8_causal_L1024-16384_paged": DecodeShape(
        "w64_b32_q8_h64kv8_causal_L1024-16384_paged", batch=32, q_len=8,
        num_q_heads=64, num_kv_heads=8, seq_len_lo=1024, seq_len_hi=16384,
        paged=True, causal=True, seed=1006),
    "w128_b16_q16_h64kv8_causal_L1024-16384_paged": DecodeShape(
        "w128_b16_q16_h64kv8_causal_L1024-16384_paged", batch=16, q_len=16,
        num_q_heads=64, num_kv_heads=8, seq_len_lo=1024, seq_len_hi=16384,
        paged=True, causal=True, seed=1007),
}
WORKLOADS.update(WIDE_WORKLOADS)

# FP8 E4M3 caches: the c2, c5 and w64 recipes with the cache quantised per tensor.
FP8_WORKLOADS = {
    "f2_b1_mha32_L131072_fp8": DecodeShape(
        "f2_b1_mha32_L131072_fp8", batch=1, q_len=1, num_q_heads=32, num_kv_heads=32,
        seq_len_lo=131072, seq_len_hi=131072, paged=False, seed=1008, kv_fp8=True),
    "f5_b32_q4_causal_h32kv8_L1024-16384_paged_fp8": DecodeShape(
        "f5_b32_q4_causal_h32kv8_L1024-16384_paged_fp8", batch=32, q_len=4,
        num_q_heads=32, num_kv_heads=8, seq_len_lo=1024, seq_len_hi=16384,
        paged=True, causal=True, seed=1009, kv_fp8=True),
    "fw64_b32_q8_h64kv8_causal_L1024-16384_paged_fp8": DecodeShape(
        "fw64_b32_q8_h64kv8_causal_L1024-16384_paged_fp8", batch=32, q_len=8,
        num_q_heads=64, num_kv_heads=8, seq_len_lo=1024, seq_len_hi=16384,
        paged=True, causal=True, seed=1010, kv_fp8=True),
}
WORKLOADS.update(FP8_WORKLOADS)


# Profiling stand-ins: the c3 recipe (same seed, length mix, paging) with 16 of
# its 64 requests (~1.1 GB of K/V instead of 4.4 GB), so a multi-pass ncu
# capture of its launch stays within a few GB of device memory; its DRAM
# traffic per launch scales to c3 by the K/V bytes.
PROFILE_WORKLOADS = {
    "c3q_b16_h32kv8_L512-32768_paged": DecodeShape(
        "c3q_b16_h32kv8_L512-32768_paged", batch=16, q_len=1, num_q_heads=32,
        num_kv_heads=8, seq_len_lo=512, seq_len_hi=32768, paged=True, seed=1003),
}
WORKLOADS.update(PROFILE_WORKLOADS)


@dataclasses.dataclass
class DecodeInputs:
    """Host (numpy) or device (torch) arrays of one workload instance.

    Layouts (all row-major, head_dim contiguous):
      q            [B, q_len, Hq, D]                 bf16 bits (uint16) / torch.bfloat16
      k_cache      paged: [P, page_size, Hkv, D]     same dtype as q, or E4M3
                   contiguous: [B, max_seq_len, Hkv, D]   bytes (uint8) with kv_fp8
      v_cache      same as k_cache
      block_table  [B, max_pages_per_seq] int32 (paged; unused slots = -1) or None
      seq_lens     [B] int32 (includes the q_len new tokens)
    """

    shape: DecodeShape
    q: object
    k_cache: object
    v_cache: object
    block_table: Optional[object]
    seq_lens: object
    max_seq_len: int
    num_pages: int           # paged: P; contiguous: 0
    page_size: int           # paged: tokens per page; contiguous: 0
    k_scale: float = 1.0     # FP8 caches: keys = k_scale * K
    v_scale: float = 1.0     # FP8 caches: values = v_scale * V

    @property
    def kv_strides(self):
        """Element strides (page-or-request, token, head) of the K/V caches."""
        _, t, h, d = self.k_cache.shape
        return (t * h * d, h * d, d)

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one call must read: every valid token of
        every request, once per KV head (K row + V row, bf16 or FP8)."""
        lens = np.asarray(_to_numpy_int(self.seq_lens), dtype=np.int64)
        s = self.shape
        return int(lens.sum()) * s.num_kv_heads * s.head_dim * 2 * kv_elem_bytes(s)


def kv_elem_bytes(shape: DecodeShape) -> int:
    return 1 if shape.kv_fp8 else 2


def quantize_e4m3(x: np.ndarray):
    """Per-tensor E4M3 quantisation of fp32 values (input preparation):
    returns (uint8 bytes, fp32 scale) with scale = max|x| / 448."""
    import torch

    amax = float(np.abs(x).max()) if x.size else 0.0
    scale = np.float32(amax / 448.0) if amax > 0 else np.float32(1.0)
    q = torch.from_numpy(np.ascontiguousarray(x / scale, dtype=np.float32))
    return q.to(torch.float8_e4m3fn).view(torch.uint8).numpy(), float(scale)


def _to_numpy_int(x):
    if isinstance(x, np.ndarray):
        return x
    return x.detach().cpu().numpy()


def draw_seq_lens(shape: DecodeShape, rng: np.random.Generator) -> np.ndarray:
    if shape.seq_len_lo == shape.seq_len_hi:
        return np.full(shape.batch, shape.seq_len_lo, dtype=np.int32)
    return rng.integers(shape.seq_len_lo, shape.seq_len_hi, size=shape.batch,
                        endpoint=True).astype(np.int32)


def draw_block_table(seq_lens: np.ndarray, page_size: int, max_pages: int,
                     rng: np.random.Generator, shuffle: bool = True,
                     extra_pages: int = 0):
    """Allocate ceil(len/page_size) physical pages per request (the block-table
    semantics of a paged KV cache) and scatter them by a random permutation of
    all physical page ids.  Returns (block_table [B, max_pages] int32 with -1
    in unused slots, num_pages)."""
    need = (seq_lens.astype(np.int64) + page_size - 1) // page_size
    total = int(need.sum()) + extra_pages
    perm = rng.permutation(total).astype(np.int32) if shuffle else \
        np.arange(total, dtype=np.int32)
    bt = np.full((len(seq_lens), max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return bt, total


def contiguous_block_table(seq_lens: np.ndarray, page_size: int, max_pages: int):
    """Identity-order block table: request b owns pages [off_b, off_b + n_b)."""
    need = (seq_lens.astype(np.int64) + page_size - 1) // page_size
    bt = np.full((len(seq_lens), max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = np.arange(off, off + n, dtype=np.int32)
        off += int(n)
    return bt, off


def _cache_dims(shape: DecodeShape, seq_lens: np.ndarray):
    max_seq_len = int(seq_lens.max()) if len(seq_lens) else 0
    if shape.paged:
        max_pages = max(1, -(-max(shape.seq_len_hi, max_seq_len) // shape.page_size))
        return max_seq_len, max_pages
    return max_seq_len, 0


def make_host_inputs(shape: DecodeShape, seed: Optional[int] = None,
                     seq_lens: Optional[np.ndarray] = None,
                     shuffle: bool = True) -> DecodeInputs:
    """Generate one workload on the host with numpy (bf16 bit patterns)."""
    rng = np.random.default_rng(shape.seed if seed is None else seed)
    if seq_lens is None:
        seq_lens = draw_seq_lens(shape, rng)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B, T, Hq, Hkv, D = (shape.batch, shape.q_len, shape.num_q_heads,
                        shape.num_kv_heads, shape.head_dim)
    max_seq_len, max_pages = _cache_dims(shape, seq_lens)
    if shape.paged:
        bt, P = draw_block_table(seq_lens, shape.page_size, max_pages, rng,
                                 shuffle=shuffle)
        kv_shape = (P, shape.page_size, Hkv, D)
    else:
        bt, P = None, 0
        kv_shape = (B, max(max_seq_len, 1), Hkv, D)
    q = rng.standard_normal((B, T, Hq, D), dtype=np.float32)
    k = rng.standard_normal(kv_shape, dtype=np.float32)
    v = rng.standard_normal(kv_shape, dtype=np.float32)
    if shape.peaked_key_fraction > 0:
        hit = rng.random(kv_shape[:3]) < shape.peaked_key_fraction
        k[hit] *= np.float32(8.0)   # exact in binary floating point
    if shape.kv_fp8:
        kb, ks = quantize_e4m3(k)
        vb, vs = quantize_e4m3(v)
        return DecodeInputs(shape, f32_to_bf16_bits(q), kb, vb, bt, seq_lens, max_seq_len,
                            P, shape.page_size if shape.paged else 0, ks, vs)
    return DecodeInputs(shape, f32_to_bf16_bits(q), f32_to_bf16_bits(k),
                        f32_to_bf16_bits(v), bt, seq_lens, max_seq_len,
                        P, shape.page_size if shape.paged else 0)


def make_device_inputs(shape: DecodeShape, seed: Optional[int] = None,
                       device: str = "cuda", seq_lens: Optional[np.ndarray] = None,
                       shuffle: bool = True) -> DecodeInputs:
    """Generate one workload directly in device memory (torch tensors).

    Lengths and block tables come from numpy (same recipe as the host path);
    q/K/V values come from torch's generator on `device`, in slabs so the fp32
    staging stays small, rounded to bf16 by torch (round to nearest even)."""
    import torch

    s = shape.seed if seed is None else seed
    rng = np.random.default_rng(s)
    if seq_lens is None:
        seq_lens = draw_seq_lens(shape, rng)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B, T, Hq, Hkv, D = (shape.batch, shape.q_len, shape.num_q_heads,
                        shape.num_kv_heads, shape.head_dim)
    max_seq_len, max_pages = _cache_dims(shape, seq_lens)
    if shape.paged:
        bt, P = draw_block_table(seq_lens, shape.page_size, max_pages, rng,
                                 shuffle=shuffle)
        kv_shape = (P, shape.page_size, Hkv, D)
    else:
        bt, P = None, 0
        kv_shape = (B, max(max_seq_len, 1), Hkv, D)
    gen = torch.Generator(device=device)
    gen.manual_seed(s)

    def normal_bf16(shp, peaked=0.0):
        out = torch.empty(shp, dtype=torch.bfloat16, device=device)
        flat = out.view(shp[0], -1)
        slab = max(1, (1 << 26) // max(1, flat.shape[1]))
        for i in range(0, shp[0], slab):
            x = torch.randn((min(slab, shp[0] - i),) + tuple(shp[1:]),
                            generator=gen, device=device, dtype=torch.float32)
            if peaked > 0:
                hit = torch.rand(x.shape[:-1], generator=gen, device=device) < peaked
                x[hit] *= 8.0
            out[i:i + x.shape[0]] = x.to(torch.bfloat16)
        return out

    def normal_e4m3(shp, seed_off, peaked=0.0):
        # two passes over the same seeded slabs: max|x| for the scale, then
        # the E4M3 bytes of x / scale (round to nearest even)
        g2 = torch.Generator(device=device)
        rows = shp[0]
        per_row = int(np.prod(shp[1:]))
        slab = max(1, (1 << 26) // max(1, per_row))

        def slabs():
            g2.manual_seed(s + seed_off)
            for i in range(0, rows, slab):
                x = torch.randn((min(slab, rows - i),) + tuple(shp[1:]), generator=g2,
                                device=device, dtype=torch.float32)
                if peaked > 0:
                    hit = torch.rand(x.shape[:-1], generator=g2, device=device) < peaked
                    x[hit] *= 8.0
                yield i, x

        amax = 0.0
        for _, x in slabs():
            amax = max(amax, float(x.abs().max()))
        scale = float(np.float32(amax / 448.0)) if amax > 0 else 1.0
        out = torch.empty(shp, dtype=torch.uint8, device=device)
        for i, x in slabs():
            out[i:i + x.shape[0]] = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
        return out, scale

    q = normal_bf16((B, T, Hq, D))
    bt_t = torch.from_numpy(bt).to(device) if bt is not None else None
    if shape.kv_fp8:
        k, ks = normal_e4m3(kv_shape, 101, shape.peaked_key_fraction)
        v, vs = normal_e4m3(kv_shape, 202)
        return DecodeInputs(shape, q, k, v, bt_t, torch.from_numpy(seq_lens).to(device),
                            max_seq_len, P, shape.page_size if shape.paged else 0, ks, vs)
    k = normal_bf16(kv_shape, shape.peaked_key_fraction)
    v = normal_bf16(kv_shape)
    return DecodeInputs(shape, q, k, v, bt_t, torch.from_numpy(seq_lens).to(device),
                        max_seq_len, P, shape.page_size if shape.paged else 0)


def small_shape(name: str = "small", batch: int = 3, q_len: int = 1,
                num_q_heads: int = 8, num_kv_heads: int = 2, lo: int = 1,
                hi: int = 300, paged: bool = True, page_size: int = 16,
                causal: bool = False, peaked: float = 0.0, seed: int = 7,
                kv_fp8: bool = False) -> DecodeShape:
    """A small workload of the same structure, for tests the oracle finishes
    in well under a second."""
    return DecodeShape(name, batch=batch, q_len=q_len, num_q_heads=num_q_heads,
                       num_kv_heads=num_kv_heads, seq_len_lo=lo, seq_len_hi=hi,
                       paged=paged, page_size=page_size, causal=causal,
                       peaked_key_fraction=peaked, seed=seed, kv_fp8=kv_fp8)
