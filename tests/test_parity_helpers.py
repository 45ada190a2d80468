"""The parity helpers' bf16 arithmetic (CPU): rounding to nearest even and
the ulp distance between bf16 values."""
import numpy as np

from tests.parity import assert_ulps_close, bf16_rne_bits, bf16_ulp_distance


def test_bf16_rounding_to_nearest_even():
    one = 0x3F80
    assert bf16_rne_bits(1.0) == one
    assert bf16_rne_bits(1.0 + 2.0 ** -8) == one          # tie: to the even neighbour
    assert bf16_rne_bits(1.0 + 3 * 2.0 ** -8) == one + 2  # tie: up to the even one
    assert bf16_rne_bits(1.0 + 2.0 ** -7) == one + 1      # exactly representable
    assert bf16_rne_bits(-2.0) == 0xC000
    assert bf16_rne_bits(0.0) == 0 and bf16_rne_bits(-0.0) == 0x8000


def test_bf16_ulp_distance():
    assert bf16_ulp_distance(0x3F80, 0x3F81) == 1
    assert bf16_ulp_distance(0x0000, 0x8000) == 0         # +0 and -0
    assert bf16_ulp_distance(0x0001, 0x8001) == 2         # smallest subnormals of both signs
    assert bf16_ulp_distance(0x3F80, 0xBF80) == 2 * 0x3F80


def test_ulps_check_ignores_small_values_and_flags_large_ones():
    ref = np.array([1.0, 0.01, -3.0])
    got = bf16_rne_bits(ref).copy()
    got[1] += 50                                          # |ref| < 0.25: not checked
    assert assert_ulps_close(got, ref) == 0
    got[2] += 3
    try:
        assert_ulps_close(got, ref)
        raise RuntimeError("not flagged")
    except AssertionError:
        pass


def test_output_tolerance_widens_only_from_four():
    """The max-abs bar is 1e-2 flat below |oracle| = 4 and 1e-2 plus half a
    bf16 ulp (2^-6 on [4, 8)) from there up."""
    from tests.parity import out_tolerance
    tol = out_tolerance(np.array([0.0, 1.5, 2.5, -3.99, 4.0, -5.0, 9.0]))
    assert np.array_equal(tol[:4], np.full(4, 1e-2))
    assert np.allclose(tol[4:], [1e-2 + 2.0 ** -6, 1e-2 + 2.0 ** -6, 1e-2 + 2.0 ** -5])
