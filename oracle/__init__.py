"""fp64 CPU oracle for split-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this package.  It shares no code with the CUDA library: the
arithmetic lives in `decode_attn_oracle.c` (plain C, fp64), built here with
gcc, and this module only marshals numpy arrays into it.

Functions
---------
decode_attention(inputs, ...)  exact softmax(q.K^T*scale).V per query head
                               ("Capstone FlashAttention", §1.1 formula; §1.2
                               three-pass safe softmax), gathered through the
                               block table (§4.1), GQA kvh = h // G (§4.2);
                               bf16 caches, or FP8 E4M3 caches with one scale
                               each (§2.2 FP8 with scaling factors).
e4m3_values()                  the 256 E4M3 codes decoded by the oracle's own
                               decoder (written from the format definition).
merge_partials(part_out, part_lse)
                               combine of normalised chunk results by their
                               log-sum-exps ("Capstone FlashAttention", §1.2
                               formal proof; §2.3 FlashDecoding reduce).
Parity status: both functions are pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_decode_attn.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math: IEEE fp64 semantics)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-pthread", "-Wall", "-Wextra", "-o", tmp, _SRC,
                           "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.oracle_decode_attn.argtypes = [
            i32, i32, i32, i32, i32, vp, vp, vp, i64, i64, i64, i32, vp, i64,
            i32, i32, i32, vp, dbl, i32, i64, i64, vp, i64, vp, vp, i32, i32, dbl, dbl]
        lib.oracle_decode_attn.restype = i32
        lib.oracle_merge_partials.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
        lib.oracle_merge_partials.restype = i32
        lib.oracle_e4m3_table.argtypes = [vp]
        lib.oracle_e4m3_table.restype = None
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     seq_lens: np.ndarray, *, num_kv_heads: int,
                     block_table: Optional[np.ndarray] = None,
                     page_size: int = 0, num_pages: int = 0,
                     scale: Optional[float] = None, causal: bool = False,
                     key_lo: int = 0, key_hi: int = 2**62,
                     rows: Optional[np.ndarray] = None,
                     threads: Optional[int] = None,
                     kv_fp8: bool = False, k_scale: float = 1.0, v_scale: float = 1.0):
    """Exact attention in fp64.

    q        uint16 bf16 bits [B, q_len, Hq, D]
    k/v      uint16 bf16 bits (or uint8 E4M3 bytes with kv_fp8: keys =
             k_scale * K, values = v_scale * V), paged [P, page_size, Hkv, D]
             (block_table given) or contiguous [B, capacity, Hkv, D]
    seq_lens int32 [B]
    rows     optional flat row ids (b*q_len + t)*Hq + h to compute
    Returns (out float64 [B, q_len, Hq, D] or [len(rows), D],
             lse float64 [B, q_len, Hq] or [len(rows)]).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    B, T, Hq, D = q.shape
    want = np.uint8 if kv_fp8 else np.uint16
    if k_cache.dtype != want or v_cache.dtype != want:
        raise TypeError("k/v caches must be bf16 bit patterns (uint16) or E4M3 bytes (uint8, kv_fp8)")
    if k_cache.shape != v_cache.shape or k_cache.shape[2] != num_kv_heads:
        raise ValueError("k/v cache shapes disagree")
    for a in (k_cache, v_cache):
        if not a.flags.c_contiguous:
            raise ValueError("oracle expects row-major caches")
    _, slots, hkv, d2 = k_cache.shape
    assert d2 == D
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if block_table is not None:
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        bt_stride, max_pages = block_table.shape[1], block_table.shape[1]
        if page_size <= 0:
            page_size = slots
        if num_pages <= 0:
            num_pages = k_cache.shape[0]
        capacity = 0
    else:
        bt_stride = max_pages = 0
        capacity = slots
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        n = len(rows)
        out = np.zeros((n, D), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
    else:
        n = B * T * Hq
        out = np.zeros((B, T, Hq, D), dtype=np.float64)
        lse = np.zeros((B, T, Hq), dtype=np.float64)
    rc = _load().oracle_decode_attn(
        B, T, Hq, num_kv_heads, D, _ptr(q), _ptr(k_cache), _ptr(v_cache),
        slots * hkv * D, hkv * D, D, page_size, _ptr(block_table), bt_stride,
        max_pages, num_pages, capacity, _ptr(seq_lens), float(scale),
        1 if causal else 0, int(key_lo), int(key_hi), _ptr(rows), n,
        _ptr(out), _ptr(lse), threads or default_threads(),
        1 if kv_fp8 else 0, float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError(f"oracle_decode_attn failed with code {rc} "
                         "(-2: block table entry out of range, -3: token beyond capacity)")
    return out, lse


def decode_attention_inputs(inp, *, rows=None, key_lo=0, key_hi=2**62,
                            threads=None):
    """Run `decode_attention` on a host `DecodeInputs` instance (numpy arrays)."""
    s = inp.shape
    return decode_attention(
        inp.q, inp.k_cache, inp.v_cache, inp.seq_lens,
        num_kv_heads=s.num_kv_heads, block_table=inp.block_table,
        page_size=inp.page_size, num_pages=inp.num_pages, scale=s.scale,
        causal=s.causal, key_lo=key_lo, key_hi=key_hi, rows=rows,
        threads=threads, kv_fp8=getattr(s, "kv_fp8", False),
        k_scale=getattr(inp, "k_scale", 1.0), v_scale=getattr(inp, "v_scale", 1.0))


def e4m3_values() -> np.ndarray:
    """float64 [256]: code c decoded by the oracle (NaN for S.1111.111)."""
    out = np.zeros(256, dtype=np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def merge_partials(part_out: np.ndarray, part_lse: np.ndarray,
                   nvalid: Optional[np.ndarray] = None):
    """Combine normalised partials [..., S, D] with log-sum-exps [..., S] into
    (out [..., D], lse [...]) in fp64.  `nvalid` limits each row to its
    leading splits."""
    part_out = np.asarray(part_out, dtype=np.float64)
    part_lse = np.asarray(part_lse, dtype=np.float64)
    lead = part_lse.shape[:-1]
    S, D = part_out.shape[-2], part_out.shape[-1]
    po = np.ascontiguousarray(part_out.reshape(-1, S, D))
    pl = np.ascontiguousarray(part_lse.reshape(-1, S))
    nrows = pl.shape[0]
    nv = None
    if nvalid is not None:
        nv = np.ascontiguousarray(np.broadcast_to(nvalid, lead).reshape(-1),
                                  dtype=np.int32)
    out = np.zeros((nrows, D), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    rc = _load().oracle_merge_partials(nrows, S, D, _ptr(po), _ptr(pl), _ptr(nv),
                                       _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_merge_partials failed with code {rc}")
    return out.reshape(lead + (D,)), lse.reshape(lead)
