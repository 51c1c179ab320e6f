"""Pins for the oracle's FP8 E4M3 codec, against facts of the OCP 8-bit float format.

Independent checks: values the format definition fixes (max normal 448, min normal
2^-6, min subnormal 2^-9, the NaN patterns), and a brute-force nearest-value search over
the 254 finite codes (a different algorithm from the encoder's binade scaling).
"""

import numpy as np
import pytest

from oracle.fp8 import e4m3_decode, e4m3_encode


def test_spec_values():
    d = e4m3_decode(np.arange(256, dtype=np.uint8))
    assert d[0x7E] == 448.0            # S.1111.110: largest finite
    assert d[0xFE] == -448.0
    assert d[0x08] == 2.0**-6          # smallest normal
    assert d[0x01] == 2.0**-9          # smallest subnormal
    assert d[0x07] == 7 * 2.0**-9      # largest subnormal
    assert d[0x38] == 1.0
    assert d[0x40] == 2.0
    assert d[0xC0] == -2.0
    assert d[0x3C] == 1.5
    assert d[0x77] == 240.0
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert d[0x00] == 0.0 and d[0x80] == 0.0 and np.signbit(d[0x80])
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0)    # monotone over the finite positive codes
    assert np.isfinite(d).sum() == 254


def _brute_force(x):
    """Nearest finite E4M3 by exhaustive search; ties to the even code; saturate."""
    codes = np.arange(0x7F, dtype=np.uint8)  # non-negative finite codes 0x00..0x7E
    vals = e4m3_decode(codes)
    out = []
    for xi in np.asarray(x, np.float64):
        a = abs(xi)
        if a >= 448.0:
            c = 0x7E
        else:
            dist = np.abs(vals - a)
            best = np.flatnonzero(dist == dist.min())
            c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
        if np.signbit(xi):
            c |= 0x80
        out.append(c)
    return np.array(out, dtype=np.uint8)


def test_encode_matches_brute_force_random():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(3000) * 50,
        rng.standard_normal(2000) * 0.01,
        rng.uniform(-500, 500, 1000),
        (rng.standard_normal(1000) * 1e-3).astype(np.float32),
    ]).astype(np.float32)
    assert np.array_equal(e4m3_encode(x), _brute_force(x))


def test_encode_ties_to_even_and_saturation():
    # midpoints between neighbours go to the even mantissa
    assert e4m3_encode(np.float32(1.0625)) == 0x38    # between 1.0 (0x38) and 1.125 (0x39)
    assert e4m3_encode(np.float32(1.1875)) == 0x3A    # between 1.125 and 1.25 (0x3A)
    assert e4m3_encode(np.float32(2.0**-10)) == 0x00  # half the smallest subnormal -> 0
    assert e4m3_encode(np.float32(3 * 2.0**-10)) == 0x02  # between 1 and 2 subnormal quanta
    assert e4m3_encode(np.float32(432.0)) == 0x7E     # between 416 and 448 -> even 448
    for big in (448.0, 449.0, 470.0, 1e6):
        assert e4m3_encode(np.float32(big)) == 0x7E
        assert e4m3_encode(np.float32(-big)) == 0xFE


@pytest.mark.parametrize("code", [c for c in range(256) if (c & 0x7F) != 0x7F])
def test_roundtrip_every_finite_code(code):
    v = e4m3_decode(np.uint8(code))
    assert e4m3_encode(np.float32(v)) == code
