"""The bf16 comparison rule of the parity tests (tests/_parity.py), checked on
hand-made values: one bf16 ulp from the oracle's rounded result passes
anywhere; two ulps fail wherever the fp32 bound 1e-4*A + 1e-6 is below one
ulp of the output, and pass near zero only when within that bound (plus
half an ulp for the final rounding); NaN matches only NaN."""
import numpy as np
import pytest

from _parity import bf16_bits_to_f64, bf16_ulp, check_bf16, near_zero


def _bits(v):
    return (np.asarray([v], np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _step(bits, n):
    return (bits.astype(np.int64) + n).astype(np.uint16)


def test_one_ulp_passes_two_fail_away_from_zero():
    y64 = np.array([1.5])
    a = np.array([10.0])                     # 1e-4 * A = 1e-3 < ulp(1.5) = 2^-7
    ref = _bits(1.5)
    assert not near_zero(ref, a).any()
    assert check_bf16(_step(ref, 1), y64, a, ref) == (0, 0)
    with pytest.raises(AssertionError):
        check_bf16(_step(ref, 2), y64, a, ref)
    with pytest.raises(AssertionError):
        check_bf16(_step(ref, -2), y64, a, ref)


def test_near_zero_outputs_are_held_to_the_fp32_bound():
    # |y| = 1e-3 with A = 100: the fp32 bound 1e-2 is many ulps of y
    y64 = np.array([1e-3])
    a = np.array([100.0])
    ref = _bits(np.float32(1e-3))
    assert near_zero(ref, a).all()
    far = _bits(np.float32(1e-3 + 5e-3))    # inside 1e-4*A + 1e-6: passes, counted strict
    strict, fail = check_bf16(far, y64, a, ref)
    assert (strict, fail) == (1, 0)
    with pytest.raises(AssertionError):     # outside the bound
        check_bf16(_bits(np.float32(1e-3 + 2e-2)), y64, a, ref)


def test_signed_zeros_are_equal_and_nan_matches_only_nan():
    y64 = np.array([0.0, np.nan])
    a = np.array([0.0, 1.0])
    ref = np.array([0x0000, 0x7FC0], np.uint16)
    assert check_bf16(np.array([0x8000, 0x7FC1], np.uint16), y64, a, ref) == (0, 0)
    with pytest.raises(AssertionError):
        check_bf16(np.array([0x0000, 0x3F80], np.uint16), y64, a, ref)


def test_ulp_spacing():
    assert bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([-3.0]))[0] == 2.0 ** -6
    assert bf16_bits_to_f64(np.array([0x3F80], np.uint16))[0] == 1.0
