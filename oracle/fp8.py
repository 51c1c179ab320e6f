"""FP8 E4M3 codec written from the OCP 8-bit floating point definition (test oracle).

E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits. Exponent field 0 encodes
subnormals m·2^-9; fields 1..15 encode (1 + m/8)·2^(e-7). There are no infinities; the
two patterns S.1111.111 are NaN, so the largest finite magnitude is 1.75·2^8 = 448.

The method stores V (pwwt.cn guide §1: "V is lowered to FP8 on Ada/Hopper") and the
softmax probabilities P in this format for the P·V product. Conversion here is
round-to-nearest-even with saturation to ±448 (the "satfinite" behaviour), which is the
conversion the method needs so that a scaled value that lands a hair above 448 is not
turned into NaN.
"""

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Decode uint8 E4M3 codes to float64 (NaN for S.1111.111)."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0**-9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((b & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_encode(x):
    """Encode real values (float32 or float64 array) to uint8 E4M3, RNE, saturating.

    The magnitude is rounded on the grid of its own binade: quantum 2^-9 below 2^-6
    (subnormals), 2^(E-3) for a normal binade [2^E, 2^(E+1)). Scaling by a power of two
    and np.rint (ties to even) are exact in float64, so the rounding is exactly RNE.
    NaN maps to 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    sat = a >= E4M3_MAX
    a_in = np.where(sat, 0.0, a)
    # binade exponent for normals; clamp to the subnormal quantum below 2^-6
    _, ex = np.frexp(np.where(a_in > 0, a_in, 1.0))  # a = f·2^ex with f in [0.5, 1)
    E = np.maximum(ex.astype(np.int64) - 1, -6)
    quantum_exp = E - 3
    q = np.rint(np.ldexp(a_in, -quantum_exp)) # integer multiple of the quantum (ties to even)
    v = np.ldexp(q, quantum_exp)              # rounded magnitude (<= 448 because a < 448)
    # bit fields from the rounded magnitude
    sub = v < 2.0**-6
    m_sub = np.rint(v * 2.0**9).astype(np.int64)
    _, ev = np.frexp(np.where(v > 0, v, 1.0))
    Ev = ev.astype(np.int64) - 1
    m_norm = np.rint((np.ldexp(v, -Ev) - 1.0) * 8.0).astype(np.int64)
    bits = np.where(sub, m_sub, ((Ev + 7) << 3) | m_norm)
    bits = np.where(sat, 0x7E, bits)  # 0.1111.110 = 448
    bits = bits | (neg.astype(np.int64) << 7)
    bits = np.where(nan, 0x7F, bits)
    return bits.astype(np.uint8)
