"""Pins for the oracle's smoothing and quantisation steps.

Independent checks: exact rational arithmetic (fractions.Fraction) for the mean,
hand-derived codes, the round-trip error bound that follows from the scale/reciprocal
definition, and the extremes (absmax -> ±127 / ±448, zero groups).
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle.fp8 import e4m3_decode
from oracle.quant import (RangeError, fixed_point_mean, fp8_channel_quant,
                          int8_group_quant, smooth)


def _nearest_f32(fr):
    """Correctly rounded float32 of an exact Fraction (ties to even), by neighbour search."""
    c = np.float32(float(fr))
    cands = [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))]
    best = min(cands, key=lambda f: (abs(Fraction(float(f)) - fr),
                                     int(np.float32(f).view(np.uint32)) & 1))
    return np.float32(best)


def test_mean_exact_rational_fp16():
    rng = np.random.default_rng(1)
    for n in (1, 2, 3, 7, 64, 129):
        x = (rng.standard_normal((n, 5)) * rng.choice([1e-3, 1, 300], (n, 5))).astype(np.float16)
        x32 = x.astype(np.float32)
        got = fixed_point_mean(x32)
        for c in range(5):
            exact = sum(Fraction(float(v)) for v in x32[:, c]) / n
            assert got[c] == _nearest_f32(exact), (n, c)


def test_mean_order_independent_and_constant():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((333, 8)).astype(np.float16).astype(np.float32)
    perm = rng.permutation(333)
    assert np.array_equal(fixed_point_mean(x).view(np.uint32),
                          fixed_point_mean(x[perm]).view(np.uint32))
    c = np.full((50, 3), np.float32(-1.25))
    assert np.all(fixed_point_mean(c) == np.float32(-1.25))


def test_mean_truncates_below_2_pow_minus_24_and_range_error():
    # bf16 can hold 2^-30; the fixed-point definition drops it (documented reading)
    x = np.full((4, 1), np.float32(2.0**-30))
    assert fixed_point_mean(x)[0] == 0.0
    n = 16
    with pytest.raises(RangeError):
        fixed_point_mean(np.full((n, 1), np.float32(2.0**38 / n)))


def test_int8_hand_case():
    # absmax 2 -> scale fl32(2/127); r = fl32(127/2) = 63.5 exactly;
    # 1*63.5 = 63.5 -> 64 (tie, even), -2*63.5 = -127, 0.5*63.5 = 31.75 -> 32,
    # 0.25*63.5 = 15.875 -> 16
    x = np.array([[1.0, -2.0, 0.5, 0.25]], dtype=np.float32)
    codes, scales = int8_group_quant(x, 1)
    assert codes.tolist() == [[64, -127, 32, 16]]
    assert scales[0] == np.float32(np.float32(2.0) / np.float32(127.0))


def test_int8_rounding_is_ties_to_even_of_the_float32_product():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((40, 16)).astype(np.float32)
    codes, scales = int8_group_quant(x, 8)
    for g in range(5):
        blk = x[g * 8:(g + 1) * 8]
        a = np.float32(np.abs(blk).max())
        r = np.float32(np.float32(127.0) / a)
        for val, code in zip(blk.ravel(), codes[g * 8:(g + 1) * 8].ravel()):
            prod = float(np.float32(val * r))
            assert code == max(-127, min(127, round(prod)))  # Python round: ties to even


@pytest.mark.parametrize("group", [1, 16, 32, 64, 128])
def test_int8_roundtrip_bound_and_extremes(group):
    rng = np.random.default_rng(group)
    n = 300
    x = (rng.standard_normal((n, 24)) * np.exp(rng.uniform(-4, 4, (n, 1)))).astype(np.float32)
    codes, scales = int8_group_quant(x, group)
    assert codes.dtype == np.int8 and np.abs(codes.astype(int)).max() <= 127
    assert len(scales) == -(-n // group)
    for g in range(len(scales)):
        blk = x[g * group:(g + 1) * group].astype(np.float64)
        cb = codes[g * group:(g + 1) * group].astype(np.float64)
        s = float(scales[g])
        a = np.abs(blk).max()
        err = np.abs(blk - cb * s)
        assert np.all(err <= s / 2 + 4 * 2.0**-24 * a)
        idx = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
        assert abs(cb[idx]) == 127


def test_int8_groups_are_independent_and_zero_group():
    x = np.ones((96, 4), np.float32)
    x[32:64] *= 1000.0
    x[64:96] = 0.0
    codes, scales = int8_group_quant(x, 32)
    assert np.all(codes[:64] == 127)           # constant groups -> all 127
    assert np.all(codes[64:] == 0) and scales[2] == 0.0
    assert scales[1] == np.float32(np.float32(1000.0) / np.float32(127.0))


def test_fp8_channel_quant_bounds_and_extremes():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((500, 12)) * np.array([1e-3, 1, 10, 1e3] * 3)).astype(np.float32)
    v[:, 11] = 0.0
    codes, scales = fp8_channel_quant(v)
    dec = e4m3_decode(codes)
    assert scales[11] == 0 and np.all(codes[:, 11] == 0)
    for c in range(11):
        s = float(scales[c])
        a = np.abs(v[:, c]).max()
        j = np.argmax(np.abs(v[:, c]))
        assert abs(dec[j, c]) == 448.0
        scaled = v[:, c].astype(np.float64) / s
        # half an ulp: 2^-4 relative for normals, 2^-10 absolute for subnormals, plus
        # the scale/reciprocal rounding (a few float32 ulps of the largest value)
        bound = np.maximum(np.abs(scaled) * 2.0**-4, 2.0**-10) + 4 * 2.0**-24 * 448
        assert np.all(np.abs(dec[:, c] - scaled) <= bound)
        assert s == np.float32(np.float32(a) / np.float32(448.0))


def test_smooth_is_one_float32_subtraction():
    x = np.array([[1.0, 2.0**-20], [3.0, -1.0]], np.float32)
    m = np.array([0.1, 2.0**-20], np.float32)
    out = smooth(x, m)
    assert out.dtype == np.float32
    assert out[0, 0] == np.float32(np.float32(1.0) - np.float32(0.1))
    assert out[0, 1] == 0.0
