"""Host-side checks of the C ABI: the library loads, exports every function the
public header declares, the parameter struct matches, and argument errors are
returned before anything touches a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from split_kv_decode_attention_gb300 import binding
from split_kv_decode_attention_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "decode_attn.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|void|char|size_t)\s*\*?\s*(decode_attn\w*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_bound_functions():
    assert declared_functions() == sorted(binding.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_params_struct_layout_matches_header(lib):
    assert ctypes.sizeof(binding.DecodeAttnParams) == 136
    p = binding.decode_attn_params_init(4, 2, 32, 8, 128, 16, 10, 100, 160, True)
    assert (p.batch, p.q_len, p.num_q_heads, p.num_kv_heads, p.head_dim) == (4, 2, 32, 8, 128)
    assert (p.page_size, p.max_pages_per_seq, p.num_pages, p.max_seq_len, p.causal) == \
        (16, 10, 100, 160, 1)
    assert abs(p.scale - 128 ** -0.5) < 1e-7
    assert (p.q_stride_batch, p.q_stride_token, p.q_stride_head) == (2 * 32 * 128, 32 * 128, 128)
    assert (p.kv_stride_page, p.kv_stride_token, p.kv_stride_head) == (16 * 8 * 128, 8 * 128, 128)
    assert p.block_table_stride == 10
    assert (p.k_scale, p.v_scale, p.flags) == (1.0, 1.0, 0)


def _call(lib, p, **kw):
    a = dict(q=16, k=16, v=16, bt=None, lens=16, out=16, lse=16, splits=1, ws=None,
             ws_bytes=0, status=None)
    a.update(kw)
    return lib.decode_attn(ctypes.byref(p), a["q"], a["k"], a["v"], a["bt"], a["lens"],
                           a["out"], a["lse"], a["splits"], a["ws"], a["ws_bytes"],
                           a["status"], None)


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 64, -3), ("num_kv_heads", 3, -2), ("q_len", 0, -2), ("batch", -1, -2),
    ("max_seq_len", -5, -2), ("flags", 4, -2)])
def test_shape_errors_are_reported_before_launch(lib, field, value, code):
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 0, 0, 0, 64, False)
    setattr(p, field, value)
    assert _call(lib, p) == code


def test_too_many_rows_rejected(lib):
    p = binding.decode_attn_params_init(1, 4, 64, 2, 128, 0, 0, 0, 64, True)  # 32 x 4 = 128 rows
    assert _call(lib, p) != -5
    p = binding.decode_attn_params_init(1, 5, 64, 2, 128, 0, 0, 0, 64, True)  # 32 x 5 = 160 rows
    assert _call(lib, p) == -5


def test_null_and_alignment_errors(lib):
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 0, 0, 0, 64, False)
    assert _call(lib, p, q=None) == -1
    assert _call(lib, p, out=None) == -1
    assert _call(lib, p, k=24) == -6           # k base not 16-byte aligned
    p.kv_stride_token = 100                     # not a multiple of 8 elements
    assert _call(lib, p) == -6


def test_fp8_cache_argument_errors(lib):
    """FP8 E4M3 caches: byte strides must be multiples of 16 and the scales
    finite; every row count up to 128 runs (both kernels read FP8)."""
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 0, 0, 0, 64, False)
    p.flags = binding.DA_FLAG_KV_FP8_E4M3
    p.kv_stride_token = 2 * 128 + 8               # a multiple of 8 but not of 16 bytes
    assert _call(lib, p) == -6
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 0, 0, 0, 64, False)
    p.flags = binding.DA_FLAG_KV_FP8_E4M3
    p.k_scale = float("inf")
    assert _call(lib, p) == -2
    p = binding.decode_attn_params_init(1, 4, 64, 8, 128, 0, 0, 0, 64, True)  # 8 x 4 = 32 rows
    p.flags = binding.DA_FLAG_KV_FP8_E4M3
    assert _call(lib, p) not in (-2, -5, -6, binding.DA_ERR_UNSUPPORTED)


def test_test_hook_flag_is_accepted(lib):
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 0, 0, 0, 64, False)
    p.flags = binding.DA_FLAG_TEST_WITHHOLD_COPY | binding.DA_FLAG_TWO_PASS
    assert _call(lib, p) != -2                    # not an unknown flag


def test_paging_errors(lib):
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 24, 4, 10, 64, False)
    assert _call(lib, p, bt=16) == -4           # page size not a multiple of 16
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 16, 4, 10, 65, False)
    assert _call(lib, p, bt=16) == -2           # 65 tokens > 4 pages x 16


def test_empty_batch_is_a_no_op(lib):
    p = binding.decode_attn_params_init(0, 1, 8, 2, 128, 0, 0, 0, 64, False)
    assert _call(lib, p, q=None, k=None, v=None, lens=None, out=None, lse=None) == 0


def test_chunk_len_and_workspace_sizes(lib):
    p = binding.decode_attn_params_init(3, 2, 8, 2, 128, 16, 100, 500, 1000, True)
    assert binding.decode_attn_chunk_len(p, 1) == 1008       # 1000 rounded up to 16
    assert binding.decode_attn_chunk_len(p, 7) == 144        # ceil(1000/7)=143 -> 144
    assert binding.decode_attn_workspace_bytes(p, 1) == 0
    rows = 3 * 2 * 8
    assert binding.decode_attn_workspace_bytes(p, 7) == rows * 7 * 129 * 4
    with pytest.raises(binding.DecodeAttnError):
        binding.decode_attn_chunk_len(p, 0)


def _call_host(lib, p, **kw):
    a = dict(q=16, k=16, v=16, bt=None, lens=16, out=16, lse=16, splits=1, ws=16,
             ws_bytes=1 << 30, status=None)
    a.update(kw)
    return lib.decode_attn_host(ctypes.byref(p), a["q"], a["k"], a["v"], a["bt"], a["lens"],
                                a["out"], a["lse"], a["splits"], a["ws"], a["ws_bytes"],
                                a["status"], None)


def test_host_entry_argument_errors(lib):
    """The host-buffer entry rejects bad arguments before it queues any copy:
    missing buffers, q / out that are not densely packed, misaligned caches,
    a workspace smaller than partials plus staging."""
    p = binding.decode_attn_params_init(2, 1, 8, 2, 128, 0, 0, 0, 64, False)
    assert _call_host(lib, p, q=None) == -1
    assert _call_host(lib, p, lse=None) == -1
    assert _call_host(lib, p, k=None) == -1
    assert _call_host(lib, p, k=24) == -6
    need = binding.decode_attn_host_workspace_bytes(p, 1)
    assert _call_host(lib, p, ws_bytes=need - 1) == -7
    assert _call_host(lib, p, ws=None) == -7
    p.q_stride_head = 256                       # heads of q not densely packed
    assert _call_host(lib, p) == -2
    p = binding.decode_attn_params_init(2, 3, 8, 2, 128, 0, 0, 0, 64, False)
    p.o_stride_batch += 128                     # padded batch rows of out
    assert _call_host(lib, p) == -2


def test_host_workspace_holds_partials_and_staging(lib):
    """decode_attn_host's workspace: decode_attn's partials, then q, out, lse,
    seq_lens, the block table and the status word at 256-byte boundaries."""
    p = binding.decode_attn_params_init(3, 2, 8, 2, 128, 16, 100, 500, 1000, True)
    rows = 3 * 2 * 8

    def r(x):
        return (x + 255) // 256 * 256
    off = r(binding.decode_attn_workspace_bytes(p, 7))
    for size in (rows * 256, rows * 256, rows * 4, 3 * 4, 3 * 100 * 4):
        off = r(off + size)
    assert binding.decode_attn_host_workspace_bytes(p, 7) == off + 16
    p1 = binding.decode_attn_params_init(3, 2, 8, 2, 128, 0, 0, 0, 1000, True)  # contiguous
    off = r(binding.decode_attn_workspace_bytes(p1, 1))
    for size in (rows * 256, rows * 256, rows * 4, 3 * 4):
        off = r(off + size)
    assert binding.decode_attn_host_workspace_bytes(p1, 1) == off + 16


def test_host_entry_empty_batch_and_no_device(lib):
    p = binding.decode_attn_params_init(0, 1, 8, 2, 128, 0, 0, 0, 64, False)
    st = ctypes.c_int32(5)
    assert _call_host(lib, p, q=None, k=None, v=None, lens=None, out=None, lse=None,
                      ws=None, status=ctypes.byref(st)) == 0
    assert st.value == 0
    import torch
    if not torch.cuda.is_available():
        p = binding.decode_attn_params_init(1, 1, 8, 2, 128, 0, 0, 0, 64, False)
        assert _call_host(lib, p) == -9          # checked before any copy is queued


def test_status_strings(lib):
    assert binding.decode_attn_status_string(0) == "ok"
    assert "128" in binding.decode_attn_status_string(-3)
    assert binding.decode_attn_status_string(-999) == "unknown status code"


def test_no_device_reported_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = binding.decode_attn_params_init(1, 1, 8, 2, 128, 0, 0, 0, 64, False)
    assert _call(lib, p) == -9
    ns, cl = ctypes.c_int32(), ctypes.c_int32()
    assert lib.decode_attn_plan(ctypes.byref(p), None, ctypes.byref(ns), ctypes.byref(cl)) == -9
