"""FP4 E2M1 codec and the two-level microscaled quantisation (test oracle).

The pages name a Blackwell variant of the method, SageAttention3, whose quantisation is "FP4
microscaling" (pwwt.cn "SageAttention deployment pitfalls guide" §5.5, API
`sageattn3_blackwell(q, k, v, is_causal=False)`), and give nothing else about it. The reading
taken here, the plainest one the rest of the method supports:

  * Elements are FP4 E2M1, the 4-bit float that FP4 tensor cores take: 1 sign bit, 2 exponent
    bits (bias 1), 1 mantissa bit. Exponent field 0 encodes the subnormals m·0.5 (0 and 0.5);
    fields 1..3 encode (1 + m/2)·2^(e-1): 1, 1.5, 2, 3, 4, 6. No infinities or NaN; 6 is the
    largest magnitude. Conversion is round-to-nearest-even with saturation to ±6.
  * "Microscaling": every block of 16 consecutive elements along the dot-product dimension
    shares one scale stored as E4M3 (the finer of the two block formats FP4 tensor cores take).
  * Two levels, as the method already has: a float32 first-level scale maps a whole token
    group (Q, K: the qk_quant_gran groups) or channel (V: over all tokens) or row (P: σ_P) onto
    [-448, 448], the E4M3 range; the block scale is then the block's largest mapped magnitude
    rounded to E4M3, and the codes are the mapped values in units of one sixth of it.

Block step, on mapped float32 values u (`microscale_blocks`):
    s_b = e4m3_rne_satfinite(max_{j in b} |u_j|)        (decoded: a multiple of 2^-9, <= 448)
    ρ_b = fl32(6 / s_b)  (0 when s_b = 0)
    c_j = e2m1_rne_satfinite(fl32(u_j · ρ_b))
    carrier_j = c_j · s_b                                (exact: at most 5 significant bits)
so that u_j ≈ carrier_j / 6. Every carrier value is a multiple of 2^-10 no larger than 2688,
hence exact in fp16; the GPU multiplies the carriers on its fp16 tensor cores and the products
and their sums are what a block-scaled FP4 product computes.
"""

import numpy as np

from .fp8 import e4m3_decode, e4m3_encode

E2M1_MAX = 6.0
BLOCK = 16          # elements per microscale block
E2M1_STEPS = 6.0    # a block's largest mapped magnitude lands on the largest E2M1 value


def e2m1_decode(codes):
    """Decode E2M1 codes (the low 4 bits of each uint8) to float64."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where((b >> 3) & 1, -1.0, 1.0)
    e = (b >> 1) & 0x3
    m = (b & 0x1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0))
    return sign * mag


def e2m1_encode(x):
    """Encode real values to E2M1 codes (uint8, low 4 bits), RNE, saturating at ±6.

    The magnitude is rounded on its binade's grid: quantum 0.5 below 2 (the subnormal 0.5 and
    the binade [1, 2) share it), 1 in [2, 4), 2 in [4, 8); np.rint rounds ties to even, which
    for these grids is the even mantissa bit. Magnitudes that round above 6 saturate to 6.
    NaN is not representable and maps to 0 with a ValueError.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("E2M1 has no NaN")
    neg = np.signbit(x)
    a = np.abs(x)
    quantum = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    v = np.rint(a / quantum) * quantum          # exact: quantum is a power of two
    v = np.minimum(v, E2M1_MAX)
    # bit fields from the rounded magnitude
    e = np.where(v < 1.0, 0, np.where(v < 2.0, 1, np.where(v < 4.0, 2, 3)))
    m = np.where(e == 0, np.rint(v * 2.0), np.rint((v / np.exp2(e - 1.0) - 1.0) * 2.0))
    bits = (e.astype(np.int64) << 1) | m.astype(np.int64)
    bits = bits | (neg.astype(np.int64) << 3)
    return bits.astype(np.uint8)


def microscale_blocks(u, axis):
    """The block step on mapped float32 values u, blocks of 16 along `axis` (the last block
    may be partial). Returns (codes uint8 E2M1 same shape, scales uint8 E4M3 with the block
    axis shortened to ceil(n / 16), carrier float64 same shape)."""
    u = np.asarray(u, dtype=np.float32)
    u = np.moveaxis(u, axis, -1)
    n = u.shape[-1]
    nb = -(-n // BLOCK)
    codes = np.zeros(u.shape, dtype=np.uint8)
    scales = np.zeros(u.shape[:-1] + (nb,), dtype=np.uint8)
    carrier = np.zeros(u.shape, dtype=np.float64)
    for b in range(nb):
        blk = u[..., b * BLOCK:(b + 1) * BLOCK]
        sb = e4m3_encode(np.max(np.abs(blk), axis=-1))
        s = e4m3_decode(sb)
        nz = s > 0
        rho = np.where(nz, (np.float32(E2M1_STEPS) / np.where(nz, s, 1.0).astype(np.float32)),
                       np.float32(0)).astype(np.float32)
        z = (blk * rho[..., None]).astype(np.float32)   # fl32(u · ρ)
        c = e2m1_encode(z)
        codes[..., b * BLOCK:(b + 1) * BLOCK] = c
        scales[..., b] = sb
        carrier[..., b * BLOCK:(b + 1) * BLOCK] = e2m1_decode(c) * s[..., None]
    return (np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis),
            np.moveaxis(carrier, -1, axis))


def fp4_group_quant(x, group):
    """Q or K' (float32 [N, d]) to two-level FP4: token groups of `group` rows share the
    first-level scale g = fl32(absmax / 448) (r = fl32(448 / absmax), u = fl32(x · r)); the
    blocks run along the channels of each row. A group whose absmax is 0 gets g = 0 and zero
    codes. Returns dict(carrier float64 [N, d], scales float32 [ceil(N / group)],
    codes, block_scales)."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    ng = -(-n // group)
    g = np.zeros(ng, dtype=np.float32)
    u = np.zeros(x.shape, dtype=np.float32)
    for i in range(ng):
        blk = x[i * group:(i + 1) * group]
        amax = np.float32(np.max(np.abs(blk))) if blk.size else np.float32(0)
        if amax == 0:
            continue
        g[i] = np.float32(amax / np.float32(448.0))
        r = np.float32(np.float32(448.0) / amax)
        u[i * group:(i + 1) * group] = (blk * r).astype(np.float32)
    codes, bs, carrier = microscale_blocks(u, axis=1)
    return dict(carrier=carrier, scales=g, codes=codes, block_scales=bs)


def fp4_channel_quant(v):
    """V' (float32 [N, d]) to two-level FP4: each channel's first-level scale is
    g_c = fl32(absmax_c / 448) over all N tokens (r_c = fl32(448 / absmax_c), as the FP8 V
    scale); the blocks run along the tokens of each channel (the P·V reduction dimension).
    Returns dict(carrier float64 [N, d], scales float32 [d], codes, block_scales)."""
    v = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v), axis=0) if v.shape[0] else np.zeros(v.shape[1], np.float32)
    amax = amax.astype(np.float32)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    g = np.where(nz, (safe / np.float32(448.0)).astype(np.float32), np.float32(0)).astype(np.float32)
    r = np.where(nz, (np.float32(448.0) / safe).astype(np.float32), np.float32(0)).astype(np.float32)
    u = (v * r[None, :]).astype(np.float32)
    codes, bs, carrier = microscale_blocks(u, axis=0)
    return dict(carrier=carrier, scales=g, codes=codes, block_scales=bs)


def fp4_p(p, sigma=448.0):
    """P (float64 probabilities, rows × keys, keys from a multiple of 16) to FP4: y =
    fl32(σ_P · p) maps the row's reference maximum to 448, then the block step along the keys.
    Returns the carrier (≈ 6 y)."""
    y = (np.asarray(p, dtype=np.float64) * sigma).astype(np.float32)
    return microscale_blocks(y, axis=-1)[2]
