"""Thin ctypes binding of libdecode_attn.so (C ABI in include/decode_attn.h).

Argument marshalling only: torch tensors supply device memory and streams,
every step of the computation runs in the library's CUDA kernels.  The names
mirror the C entry points.  There is no fallback: if the library is missing or
no GPU is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libdecode_attn.so")

HEAD_DIM = 128
MAX_ROWS = 128
TOKEN_TILE = 16

DA_OK = 0
DA_STATUS_BAD_PAGE = 1
DA_STATUS_SEQ_LEN = 2
DA_STATUS_SHORT_CAUSAL = 4
DA_STATUS_TIMEOUT = 8
DA_FLAG_TWO_PASS = 1
DA_FLAG_KV_FP8_E4M3 = 2
DA_FLAG_TEST_WITHHOLD_COPY = 0x100
DA_ERR_UNSUPPORTED = -12

EXPORTED_SYMBOLS = (
    "decode_attn_params_init", "decode_attn_plan", "decode_attn_plan_slots", "decode_attn_chunk_len",
    "decode_attn_workspace_bytes", "decode_attn", "decode_attn_split", "decode_attn_combine",
    "decode_attn_status_string", "decode_attn_launch_count", "decode_attn_static_workspace",
    "decode_attn_host_workspace_bytes", "decode_attn_host", "decode_attn_device_plan",
)
DA_ERR_STATIC_WORKSPACE_LIMIT = -11
STATIC_WORKSPACE_BYTES = 16 << 20


class DecodeAttnParams(ctypes.Structure):
    """Mirror of `decode_attn_params` (same field order and types)."""

    _fields_ = [
        ("batch", ctypes.c_int32), ("q_len", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32), ("causal", ctypes.c_int32),
        ("scale", ctypes.c_float), ("flags", ctypes.c_int32),
        ("q_stride_batch", ctypes.c_int64), ("q_stride_token", ctypes.c_int64),
        ("q_stride_head", ctypes.c_int64), ("o_stride_batch", ctypes.c_int64),
        ("o_stride_token", ctypes.c_int64), ("o_stride_head", ctypes.c_int64),
        ("kv_stride_page", ctypes.c_int64), ("kv_stride_token", ctypes.c_int64),
        ("kv_stride_head", ctypes.c_int64), ("block_table_stride", ctypes.c_int64),
        ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
    ]


class DecodeAttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where} failed: {decode_attn_status_string(code)} (code {code})")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(DecodeAttnParams)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        pi32 = ctypes.POINTER(ctypes.c_int32)
        L.decode_attn_params_init.argtypes = [P] + [i32] * 10
        L.decode_attn_params_init.restype = None
        L.decode_attn_plan.argtypes = [P, vp, pi32, pi32]
        L.decode_attn_plan_slots.argtypes = [P, vp, ctypes.c_int64, pi32, pi32]
        L.decode_attn_chunk_len.argtypes = [P, i32, pi32]
        L.decode_attn_workspace_bytes.argtypes = [P, i32, ctypes.POINTER(sz)]
        L.decode_attn.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp, vp]
        L.decode_attn_split.argtypes = L.decode_attn.argtypes
        L.decode_attn_static_workspace.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp]
        L.decode_attn_combine.argtypes = [P, vp, i32, i32, vp, sz, vp, vp, vp]
        L.decode_attn_status_string.argtypes = [ctypes.c_int]
        L.decode_attn_status_string.restype = ctypes.c_char_p
        L.decode_attn_launch_count.argtypes = [P, i32]
        L.decode_attn_host_workspace_bytes.argtypes = [P, i32, ctypes.POINTER(sz)]
        L.decode_attn_host.argtypes = L.decode_attn.argtypes
        L.decode_attn_device_plan.argtypes = [P, vp, vp, sz, vp, vp]
        for f in ("decode_attn_plan", "decode_attn_plan_slots", "decode_attn_chunk_len",
                  "decode_attn_workspace_bytes",
                  "decode_attn", "decode_attn_split", "decode_attn_combine",
                  "decode_attn_launch_count", "decode_attn_static_workspace",
                  "decode_attn_host_workspace_bytes", "decode_attn_host",
                  "decode_attn_device_plan"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def decode_attn_status_string(code: int) -> str:
    return lib().decode_attn_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != DA_OK:
        raise DecodeAttnError(code, where)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def decode_attn_params_init(batch: int, q_len: int, num_q_heads: int, num_kv_heads: int,
                            head_dim: int = HEAD_DIM, page_size: int = 0,
                            max_pages_per_seq: int = 0, num_pages: int = 0,
                            max_seq_len: int = 0, causal: bool = False) -> DecodeAttnParams:
    p = DecodeAttnParams()
    lib().decode_attn_params_init(ctypes.byref(p), batch, q_len, num_q_heads, num_kv_heads,
                                  head_dim, page_size, max_pages_per_seq, num_pages,
                                  max_seq_len, 1 if causal else 0)
    return p


def params_from_tensors(q, k_cache, block_table=None, *, max_seq_len: int,
                        causal: bool = False, scale: Optional[float] = None,
                        out=None, two_pass: bool = False, k_scale: float = 1.0,
                        v_scale: float = 1.0) -> DecodeAttnParams:
    """Describe torch tensors: q/out [B, q_len, Hq, D]; k_cache paged
    [P, page_size, Hkv, D] (block_table [B, max_pages] given) or contiguous
    [B, S, Hkv, D].  Strides are taken from the tensors.  A one-byte cache
    (uint8 or float8_e4m3fn) is an FP8 E4M3 cache with the given scales."""
    B, T, Hq, D = q.shape
    n0, n1, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_cache differ")
    p = DecodeAttnParams()
    p.batch, p.q_len, p.num_q_heads, p.num_kv_heads, p.head_dim = B, T, Hq, Hkv, D
    p.max_seq_len = int(max_seq_len)
    p.causal = 1 if causal else 0
    p.flags = DA_FLAG_TWO_PASS if two_pass else 0
    if k_cache.element_size() == 1:
        p.flags |= DA_FLAG_KV_FP8_E4M3
    p.k_scale, p.v_scale = float(k_scale), float(v_scale)
    p.scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    p.q_stride_batch, p.q_stride_token, p.q_stride_head = (int(s) for s in q.stride()[:3])
    o = out if out is not None else q
    p.o_stride_batch, p.o_stride_token, p.o_stride_head = (int(s) for s in o.stride()[:3])
    p.kv_stride_page, p.kv_stride_token, p.kv_stride_head = (int(s) for s in k_cache.stride()[:3])
    if block_table is not None:
        p.page_size = n1
        p.num_pages = n0
        p.max_pages_per_seq = block_table.shape[1]
        p.block_table_stride = int(block_table.stride(0))
    return p


def decode_attn_plan(p: DecodeAttnParams, host_seq_lens=None) -> Tuple[int, int]:
    import numpy as np
    ns, cl = ctypes.c_int32(), ctypes.c_int32()
    arr = None
    if host_seq_lens is not None:
        arr = np.ascontiguousarray(host_seq_lens, dtype=np.int32)
    _check(lib().decode_attn_plan(ctypes.byref(p),
                                  None if arr is None else arr.ctypes.data,
                                  ctypes.byref(ns), ctypes.byref(cl)), "decode_attn_plan")
    return ns.value, cl.value


def decode_attn_plan_slots(p: DecodeAttnParams, host_seq_lens, resident_ctas: int) -> Tuple[int, int]:
    """The planner for an explicit number of resident split CTAs (host only)."""
    import numpy as np
    ns, cl = ctypes.c_int32(), ctypes.c_int32()
    arr = None
    if host_seq_lens is not None:
        arr = np.ascontiguousarray(host_seq_lens, dtype=np.int32)
    _check(lib().decode_attn_plan_slots(ctypes.byref(p),
                                        None if arr is None else arr.ctypes.data,
                                        int(resident_ctas), ctypes.byref(ns), ctypes.byref(cl)),
           "decode_attn_plan_slots")
    return ns.value, cl.value


def decode_attn_chunk_len(p: DecodeAttnParams, num_splits: int) -> int:
    c = ctypes.c_int32()
    _check(lib().decode_attn_chunk_len(ctypes.byref(p), int(num_splits), ctypes.byref(c)),
           "decode_attn_chunk_len")
    return c.value


def decode_attn_workspace_bytes(p: DecodeAttnParams, num_splits: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().decode_attn_workspace_bytes(ctypes.byref(p), int(num_splits), ctypes.byref(n)),
           "decode_attn_workspace_bytes")
    return n.value


def decode_attn_launch_count(p: DecodeAttnParams, num_splits: int) -> int:
    n = lib().decode_attn_launch_count(ctypes.byref(p), int(num_splits))
    if n < 0:
        raise DecodeAttnError(n, "decode_attn_launch_count")
    return n


def decode_attn(q, k_cache, v_cache, block_table, seq_lens, *, max_seq_len: int,
                causal: bool = False, scale: Optional[float] = None, num_splits: int = 0,
                out=None, lse=None, workspace=None, status=None, stream=None,
                params: Optional[DecodeAttnParams] = None, two_pass: bool = False,
                k_scale: float = 1.0, v_scale: float = 1.0):
    """Run decode attention; returns (out bf16 [B, q_len, Hq, D], lse fp32
    [B, q_len, Hq]).  Output, LSE and workspace tensors are allocated with
    torch when not given; `num_splits <= 0` lets the library's planner choose
    (on the device, from the lengths in `seq_lens`, for two or more requests)."""
    import torch

    B, T, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, T, Hq), dtype=torch.float32, device=q.device)
    p = params if params is not None else params_from_tensors(
        q, k_cache, block_table, max_seq_len=max_seq_len, causal=causal, scale=scale, out=out,
        two_pass=two_pass, k_scale=k_scale, v_scale=v_scale)
    num_splits = max(0, int(num_splits))
    need = decode_attn_workspace_bytes(p, num_splits)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty((need + 15) // 16 * 4, dtype=torch.float32, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().decode_attn(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                             _ptr(block_table), _ptr(seq_lens), _ptr(out), _ptr(lse),
                             int(num_splits), _ptr(workspace) if need > 0 else None, ws_bytes,
                             _ptr(status), _stream_handle(stream)), "decode_attn")
    return out, lse


def decode_attn_host_workspace_bytes(p: DecodeAttnParams, num_splits: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().decode_attn_host_workspace_bytes(ctypes.byref(p), int(num_splits),
                                                  ctypes.byref(n)),
           "decode_attn_host_workspace_bytes")
    return n.value


def decode_attn_host(q_host, k_cache, v_cache, block_table_host, seq_lens_host, *,
                     max_seq_len: int, causal: bool = False, scale: Optional[float] = None,
                     num_splits: int = 0, out_host=None, lse_host=None, workspace=None,
                     stream=None, params: Optional[DecodeAttnParams] = None,
                     two_pass: bool = False, k_scale: float = 1.0, v_scale: float = 1.0):
    """decode_attn with q, block table and seq_lens in host memory (torch CPU
    tensors, ideally pinned) and out / lse returned to host memory; the K/V
    cache stays on the device.  One C call: with pinned buffers the kernels
    read and write them in place, otherwise copies in and out; the stream is
    synchronised.  Returns (out_host, lse_host, status bits)."""
    import numpy as np
    import torch

    B, T, Hq, D = q_host.shape
    if out_host is None:
        out_host = torch.empty((B, T, Hq, D), dtype=torch.bfloat16).pin_memory()
    if lse_host is None:
        lse_host = torch.empty((B, T, Hq), dtype=torch.float32).pin_memory()
    p = params if params is not None else params_from_tensors(
        q_host, k_cache, block_table_host, max_seq_len=max_seq_len, causal=causal, scale=scale,
        out=out_host, two_pass=two_pass, k_scale=k_scale, v_scale=v_scale)
    if workspace is None:   # (a given workspace is checked by the C call itself)
        if num_splits <= 0:  # the library's planner, with the actual lengths
            num_splits, _ = decode_attn_plan(p, np.asarray(seq_lens_host, dtype=np.int32))
        need = decode_attn_host_workspace_bytes(p, num_splits)
        workspace = torch.empty((need + 15) // 16 * 4, dtype=torch.float32, device=k_cache.device)
    global _host_status
    if _host_status is None:   # a page-locked word: the kernels write it in place
        _host_status = torch.zeros(1, dtype=torch.int32).pin_memory()
    status_ptr = _host_status.data_ptr()
    _check(lib().decode_attn_host(ctypes.byref(p), _ptr(q_host), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(block_table_host), _ptr(seq_lens_host), _ptr(out_host),
                                  _ptr(lse_host), int(num_splits), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  status_ptr, _stream_handle(stream)),
           "decode_attn_host")
    return out_host, lse_host, ctypes.c_int32.from_address(status_ptr).value


_host_status = None


def decode_attn_device_plan(p: DecodeAttnParams, seq_lens, workspace, status=None, stream=None):
    """Run the device planner alone (the first launch of a device-planned
    decode_attn call) into `workspace`; read the plan back with
    device_plan_view()."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().decode_attn_device_plan(ctypes.byref(p), _ptr(seq_lens), _ptr(workspace),
                                         ws_bytes, _ptr(status), _stream_handle(stream)),
           "decode_attn_device_plan")


def device_plan_view(workspace, p: DecodeAttnParams):
    """(plan int32[4] = chunk_len, items, chunks of the longest request,
    capacity; pre int32[B + 1]; items int32[capacity, 4] = (b, kv head, chunk,
    length)) views of a device-planned call's workspace, per the layout in the
    header."""
    import torch
    b = workspace.view(-1).view(torch.int32)

    def r256(x):
        return (x + 255) // 256 * 256

    plan = b[:4]
    off = 256
    pre = b[off // 4: off // 4 + p.batch + 1]
    off = r256(off + (p.batch + 1) * 4)
    cap = int(plan[3].item())
    items = b[off // 4: off // 4 + 4 * cap].view(cap, 4)
    return plan, pre, items


def decode_attn_combine(p: DecodeAttnParams, seq_lens, num_splits: int, chunk_len: int,
                        workspace, out, lse, stream=None):
    """Merge the partials held in `workspace` into out/lse (rows of requests
    spanning two or more chunks); num_splits <= 0 after a device-planned
    split pass."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().decode_attn_combine(ctypes.byref(p), _ptr(seq_lens), int(num_splits),
                                     int(chunk_len), _ptr(workspace), ws_bytes, _ptr(out),
                                     _ptr(lse), _stream_handle(stream)), "decode_attn_combine")
    return out, lse


def workspace_views(workspace, p: DecodeAttnParams, num_splits: int):
    """(part_o [B, q_len, Hq, S, D], part_lse [B, q_len, Hq, S]) views of a
    workspace tensor, per the layout documented for decode_attn_workspace_bytes."""
    S = num_splits
    rows = p.batch * p.q_len * p.num_q_heads
    f = workspace.view(-1)[: rows * S * (HEAD_DIM + 1)]
    po = f[: rows * S * HEAD_DIM].view(p.batch, p.q_len, p.num_q_heads, S, HEAD_DIM)
    pl = f[rows * S * HEAD_DIM:].view(p.batch, p.q_len, p.num_q_heads, S)
    return po, pl


def decode_attn_split(p: DecodeAttnParams, q, k_cache, v_cache, block_table, seq_lens, out,
                      lse, num_splits: int, workspace=None, status=None, stream=None):
    """The split pass alone (same arguments as the C entry point): final
    out/lse for requests that fit one chunk, partials in `workspace` for the
    rest; decode_attn_combine() with the same num_splits finishes them."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().decode_attn_split(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(block_table), _ptr(seq_lens), _ptr(out), _ptr(lse),
                                   int(num_splits), _ptr(workspace), ws_bytes, _ptr(status),
                                   _stream_handle(stream)), "decode_attn_split")
    return out, lse


def decode_attn_static_workspace(p: DecodeAttnParams, q, k_cache, v_cache, block_table,
                                 seq_lens, out, lse, num_splits: int = 0, status=None,
                                 stream=None):
    """decode_attn() without a caller workspace, for callers that cannot
    allocate device memory: the partials live in the library's fixed 16 MiB
    device array (shared by all calls on a device; overlapping calls race).
    Raises DecodeAttnError(-11) when a call needs more than that."""
    _check(lib().decode_attn_static_workspace(
        ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(out), _ptr(lse), int(num_splits), _ptr(status),
        _stream_handle(stream)), "decode_attn_static_workspace")
    return out, lse
