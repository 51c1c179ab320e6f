"""Stage 1 and 2 of the method: smoothing and quantisation (test oracle).

Follows pwwt.cn "SageAttention deployment pitfalls guide":
  §1   Q and K go to INT8 with fine-grained ("per-block / per-thread") scale factors,
       V goes to FP8;
  §4.2 smooth_k subtracts K's mean along the sequence dimension; smooth_v does the same
       for V; qk_quant_gran selects per_warp / per_thread granularity;
and pnsm.cn "SageAttention on AMD 9070 XT without the HIP SDK" §2 (split into small
blocks, take each block's range, compress to 8 bits).

The pages give no group sizes, rounding rule or summation order. The readings taken here:
token groups of 128/32/1 rows for Q and 64/64/16 rows for K (per_block / per_warp /
per_thread), restarting per sequence; scale = absmax/127 with codes from a reciprocal
multiply and ties-to-even rounding; an order-free fixed-point mean. Everything is per
(batch, head) — or per (sequence, head) for varlen.
"""

import numpy as np

from .fp8 import e4m3_encode

# token-group sizes per granularity, for Q and for K
GRAN_PER_BLOCK, GRAN_PER_WARP, GRAN_PER_THREAD = 0, 1, 2
Q_GROUP = {GRAN_PER_BLOCK: 128, GRAN_PER_WARP: 32, GRAN_PER_THREAD: 1}
K_GROUP = {GRAN_PER_BLOCK: 64, GRAN_PER_WARP: 64, GRAN_PER_THREAD: 16}

FIXED_POINT_BITS = 24  # every fp16 value is an integer multiple of 2^-24


class RangeError(ValueError):
    """An input too large for the exact fixed-point mean."""


def fixed_point_mean(x):
    """Mean over axis 0 of a float32 [N, d] array, defined to be order-independent.

    S_c = sum_j trunc(x_jc * 2^24) in int64 (exact: x * 2^24 is exact in float64, and for
    fp16 inputs the truncation drops nothing); mean_c = fl32(fl64(fl64(S_c) * 2^-24 / N)).
    Inputs with |x| >= 2^38 / N could overflow int64 and raise RangeError.
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    if n == 0:
        raise ValueError("mean over an empty sequence")
    limit = 2.0 ** (62 - FIXED_POINT_BITS) / n
    if np.any(np.abs(x.astype(np.float64)) >= limit):
        raise RangeError("input magnitude too large for the fixed-point mean")
    fixed = np.trunc(x.astype(np.float64) * 2.0**FIXED_POINT_BITS).astype(np.int64)
    s = fixed.sum(axis=0, dtype=np.int64)
    return (s.astype(np.float64) * 2.0**-FIXED_POINT_BITS / np.float64(n)).astype(np.float32)


def int8_group_quant(x, group):
    """Symmetric INT8 quantisation of float32 [N, d] rows in groups of `group` tokens.

    For each group: absmax = max |x| (float32), scale = fl32(absmax / 127),
    r = fl32(127 / absmax), code = clamp(rint_even(fl32(x * r)), -127, 127).
    A group whose absmax is 0 gets scale 0 and all-zero codes. The last group may be
    partial. Returns (codes int8 [N, d], scales float32 [ceil(N / group)]).
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    ng = -(-n // group)
    codes = np.zeros(x.shape, dtype=np.int8)
    scales = np.zeros(ng, dtype=np.float32)
    for g in range(ng):
        blk = x[g * group:(g + 1) * group]
        amax = np.float32(np.max(np.abs(blk))) if blk.size else np.float32(0)
        if amax == 0:
            continue
        scales[g] = np.float32(amax / np.float32(127.0))
        r = np.float32(np.float32(127.0) / amax)
        q = np.rint(blk * r)  # float32 product, then ties-to-even
        codes[g * group:(g + 1) * group] = np.clip(q, -127, 127).astype(np.int8)
    return codes, scales


def fp8_channel_quant(v):
    """Per-channel FP8 E4M3 quantisation of float32 [N, d] (scale over all N tokens).

    absmax_c = max_j |v_jc|, scale_c = fl32(absmax_c / 448), r_c = fl32(448 / absmax_c),
    code = e4m3_rne_satfinite(fl32(v * r_c)). A channel with absmax 0 gets scale 0 and
    zero codes. Returns (codes uint8 [N, d], scales float32 [d]).
    """
    v = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v), axis=0) if v.shape[0] else np.zeros(v.shape[1], np.float32)
    amax = amax.astype(np.float32)
    nz = amax > 0
    safe = np.where(nz, amax, np.float32(1.0)).astype(np.float32)
    scales = np.where(nz, (safe / np.float32(448.0)).astype(np.float32), np.float32(0)).astype(np.float32)
    r = np.where(nz, (np.float32(448.0) / safe).astype(np.float32), np.float32(0)).astype(np.float32)
    scaled = (v * r[None, :]).astype(np.float32)
    return e4m3_encode(scaled), scales


def smooth(x, mean):
    """x - mean, one float32 subtraction per element (§4.2 smooth_k / smooth_v)."""
    return (np.asarray(x, np.float32) - np.asarray(mean, np.float32)[None, :]).astype(np.float32)
