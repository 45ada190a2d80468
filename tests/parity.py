"""Shared helpers of the parity tests: device upload and the tolerance rule.

Tolerance (fixed for this path): bf16 outputs within max-abs 1e-2 and
mean-abs 1e-3 of the fp64 oracle, fp32 LSE within abs 1e-3; the parity tests
(fixed, random and full-size cases) also bound the distance in bf16 ulps to
the rounded oracle where |oracle| >= 0.25.  One refinement, and only one:
where |oracle| >= 4 the bf16 output grid itself is coarser than the bar (half
an ulp of bf16 on [4, 8) is 2^-6 ~ 0.0156 > 1e-2), so there an element may
also be off by half a bf16 ulp of the oracle value on top of the 1e-2.
Below 4 the bar is 1e-2 flat (half an ulp is 2^-8 ~ 0.0039 on [1, 2) and
2^-7 ~ 0.0078 on [2, 4), inside the bar).
"""
import numpy as np

OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) around |x|."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0**-126)))
    return 0.5 * np.exp2(e - 7)


def out_tolerance(ref: np.ndarray) -> np.ndarray:
    ref = np.asarray(ref, dtype=np.float64)
    return np.where(np.abs(ref) >= 4.0, OUT_MAX_ABS + bf16_half_ulp(ref), OUT_MAX_ABS)


def assert_out_close(got, ref, what="out"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    tol = out_tolerance(ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements beyond tolerance; worst at {i}: "
                             f"got {got[i]}, oracle {ref[i]}, |err| {err[i]:.3e}")
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean abs error {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def assert_lse_close(got, ref, what="lse"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern differs"
    if (~ninf).any():
        err = np.abs(got[~ninf] - ref[~ninf])
        assert err.max() <= LSE_MAX_ABS, f"{what}: max abs error {err.max():.3e}"
        return float(err.max())
    return 0.0


def bf16_rne_bits(x) -> np.ndarray:
    """bf16 bit patterns of x rounded to nearest even (through fp32)."""
    f = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_ulp_distance(a_bits, b_bits) -> np.ndarray:
    """Number of bf16 values between two bf16 bit patterns (+0 and -0 equal)."""
    def line(b):
        b = np.asarray(b).astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(line(a_bits) - line(b_bits))


# Where |oracle| >= ULP_MIN_ABS, the output is within ULP_MAX bf16 ulps of the
# oracle rounded to bf16 (near zero the ulp shrinks and the absolute bar is
# the meaningful one)
ULP_MIN_ABS = 0.25
ULP_MAX = 2


def assert_ulps_close(got_bits, ref, what="out"):
    ref = np.asarray(ref, dtype=np.float64).ravel()
    d = bf16_ulp_distance(np.asarray(got_bits).ravel(), bf16_rne_bits(ref))
    sel = np.abs(ref) >= ULP_MIN_ABS
    if sel.any():
        worst = int(d[sel].max())
        assert worst <= ULP_MAX, f"{what}: {worst} bf16 ulps from the rounded oracle"
        return worst
    return 0


def to_device(inp, device="cuda"):
    """Upload a host DecodeInputs (numpy bf16 bits, FP8 caches as bytes) to
    torch device tensors."""
    import torch

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).to(device)

    def kv(a):  # bf16 bits, or FP8 E4M3 bytes as uint8
        if a.dtype == np.uint8:
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)
        return bf(a)

    bt = None if inp.block_table is None else torch.from_numpy(inp.block_table).to(device)
    return (bf(inp.q), kv(inp.k_cache), kv(inp.v_cache), bt,
            torch.from_numpy(np.ascontiguousarray(inp.seq_lens)).to(device))


def bf16_tensor_to_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_tensor_to_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
