"""Split-KV decode attention (Flash-Decoding) for GB300 (sm_103a).

The compute path lives in the CUDA library `libdecode_attn.so` built from
`csrc/` (C ABI declared in `include/decode_attn.h`); `binding` marshals torch
tensors into it.  The library is loaded on first use and every entry point
raises if it is missing: there is no CPU fallback.
"""
from . import workloads  # noqa: F401  (input generation only)

__all__ = ["workloads"]
