"""Pins for the oracle's FP4 microscaled variant (oracle/fp4.py and attention pv="fp4").

The E2M1 codec is checked against the format's definition (a value table written from the
field layout, and a brute-force nearest-value search with ties to the even mantissa); the block
step against its defining properties; the attention mode against closed forms on inputs that
FP4 represents exactly, so that every scale factor of the variant (g/6 per operand, σ_P = 2688)
shows up in an exact result.
"""

import numpy as np
import pytest

from oracle.attention import ACC_FP32, attention_fp64, sage_attention
from oracle.fp4 import (BLOCK, e2m1_decode, e2m1_encode, fp4_channel_quant, fp4_group_quant,
                        fp4_p, microscale_blocks)
from oracle.fp8 import e4m3_decode, e4m3_encode
from oracle.quant import GRAN_PER_BLOCK, GRAN_PER_THREAD, GRAN_PER_WARP

# E2M1 magnitudes by (exponent field, mantissa bit), from the definition: field 0 holds the
# subnormals m * 0.5, fields 1..3 the normals (1 + m/2) * 2^(e - 1)
TABLE = {(0, 0): 0.0, (0, 1): 0.5, (1, 0): 1.0, (1, 1): 1.5, (2, 0): 2.0, (2, 1): 3.0,
         (3, 0): 4.0, (3, 1): 6.0}


def test_e2m1_decode_table():
    for code in range(16):
        e, m, neg = (code >> 1) & 3, code & 1, code >> 3
        want = -TABLE[(e, m)] if neg else TABLE[(e, m)]
        got = e2m1_decode(np.uint8(code))
        assert got == want and np.signbit(got) == bool(neg)


def _nearest_even(x):
    """Brute force: the representable magnitude nearest |x| (ties: even mantissa bit), or 6
    beyond the largest; the sign carried over."""
    mags = sorted({(v, m) for (e, m), v in TABLE.items()})
    a = abs(x)
    if a >= 6.0:
        best = 6.0
    else:
        dist = [(abs(a - v), m, v) for v, m in mags]
        dmin = min(d for d, _, _ in dist)
        cands = [(m, v) for d, m, v in dist if d == dmin]
        best = min(cands)[1]   # mantissa bit 0 first
    return -best if np.signbit(x) else best


def test_e2m1_encode_brute_force():
    grid = np.arange(-8.0, 8.0 + 1e-9, 1.0 / 64.0)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 6.5, 100.0, 1e30])
    x = np.concatenate([grid, ties, -ties, np.nextafter(ties, 0), np.nextafter(ties, 10)])
    got = e2m1_decode(e2m1_encode(x))
    want = np.array([_nearest_even(v) for v in x])
    np.testing.assert_array_equal(got, want)
    # ties resolve to the even mantissa: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2,
    # 2.5 -> 2, 3.5 -> 4, 5 -> 4
    np.testing.assert_array_equal(e2m1_decode(e2m1_encode(ties[:7])), [0, 1, 1, 2, 2, 4, 4])


def test_e2m1_round_trip_and_errors():
    codes = np.arange(16, dtype=np.uint8)
    np.testing.assert_array_equal(e2m1_encode(e2m1_decode(codes)), codes)
    with pytest.raises(ValueError):
        e2m1_encode(np.array([np.nan]))


def test_block_step_properties():
    rng = np.random.default_rng(0)
    u = (rng.standard_normal((37, 50)) * np.exp(rng.uniform(-6, 6, (37, 1)))).astype(np.float32)
    codes, bs, car = microscale_blocks(u, axis=1)
    assert bs.shape == (37, 4)        # 50 channels: 3 full blocks and one of 2
    s = e4m3_decode(bs)
    for b in range(4):
        blk = u[:, b * BLOCK:(b + 1) * BLOCK]
        # the scale is the block's largest magnitude rounded to E4M3
        np.testing.assert_array_equal(bs[:, b], e4m3_encode(np.abs(blk).max(axis=1)))
        rho = (np.float32(6.0) / s[:, b].astype(np.float32)).astype(np.float32)
        z = (blk * rho[:, None]).astype(np.float32)
        c = e2m1_decode(codes[:, b * BLOCK:(b + 1) * BLOCK])
        # each code is z rounded to the E2M1 grid: within half a grid step (saturating at 6)
        half = np.where(np.abs(z) < 2, 0.25, np.where(np.abs(z) < 4, 0.5, 1.0))
        assert np.all(np.abs(np.clip(z, -6, 6) - c) <= half)
        # the largest magnitude of every block lands on ±6
        imax = np.abs(blk).argmax(axis=1)
        assert np.all(np.abs(c[np.arange(37), imax]) == 6.0)
        # the carrier is code x scale, exact in fp16 (a multiple of 2^-10, at most 2688)
        cb = car[:, b * BLOCK:(b + 1) * BLOCK]
        np.testing.assert_array_equal(cb, c * s[:, b][:, None])
        assert np.all(np.abs(cb) <= 2688) and np.all(cb * 1024 == np.rint(cb * 1024))


def test_block_step_hand_case():
    # scale 384 = 1.5 * 2^8 (an E4M3 value), so rho = 6 / 384 = 2^-6 exactly and every
    # u = 64 c (c an E2M1 value) is reproduced exactly; 80 = 64 * 1.25 ties to 1 (even), 224 =
    # 64 * 3.5 ties to 4; 0.5 * 64 = 32
    u = np.float32([[384, 64, 96, 128, 192, 256, -32, 0, 80, 224, -384, 1, 2, 3, 4, 5]])
    codes, bs, car = microscale_blocks(u, axis=1)
    assert e4m3_decode(bs)[0, 0] == 384.0
    want_c = [6, 1, 1.5, 2, 3, 4, -0.5, 0, 1, 4, -6, 0, 0, 0, 0, 0]
    np.testing.assert_array_equal(e2m1_decode(codes)[0], want_c)
    np.testing.assert_array_equal(car[0], np.array(want_c) * 384.0)


def test_zero_block_and_zero_group():
    codes, bs, car = microscale_blocks(np.zeros((2, 16), np.float32), axis=1)
    assert not codes.any() and not bs.any() and not car.any()
    q = fp4_group_quant(np.zeros((5, 16), np.float32), 2)
    assert not q["scales"].any() and not q["carrier"].any()


def test_group_quant_reconstruction_bound():
    # x ≈ g · carrier / 6 within half an E2M1 step of the block scale, plus the first-level
    # mapping's float32 rounding
    rng = np.random.default_rng(1)
    x = rng.standard_normal((70, 40)).astype(np.float32) * 3
    for group in (1, 16, 32, 64):
        q = fp4_group_quant(x, group)
        g = np.repeat(q["scales"], group)[:70].astype(np.float64)
        s = np.repeat(e4m3_decode(q["block_scales"]), BLOCK, axis=1)[:, :40]
        xhat = g[:, None] * q["carrier"] / 6.0
        bound = g[:, None] * s / 6.0 * 1.0 + 1e-5 * np.abs(x)
        assert np.all(np.abs(x - xhat) <= bound)
        # the group's largest magnitude is reproduced to its E4M3 scale's rounding
        for i in range(-(-70 // group)):
            blk = x[i * group:(i + 1) * group]
            assert q["scales"][i] == np.float32(np.abs(blk).max() / np.float32(448))


def test_channel_quant_blocks_run_along_tokens():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((40, 3)).astype(np.float32)
    v[17, 1] = 50.0           # one outlier: only block 1 of channel 1 loses resolution
    q = fp4_channel_quant(v)
    assert q["block_scales"].shape == (3, 3)   # 40 tokens -> blocks of 16, 16, 8 per channel
    assert q["scales"][1] == np.float32(np.float32(50.0) / np.float32(448.0))
    bs = e4m3_decode(q["block_scales"])
    assert bs[1, 1] == 448.0 and bs[0, 1] < 448.0 / 4


def _lossless_rows(rng, n, d):
    """Rows that two-level FP4 reproduces exactly: each 16-channel block holds E2M1 values
    with largest magnitude 6 (block scale 384 after the group maps the row maximum 7 to
    448), and channel 0 holds the group maximum ±7 alone in its block."""
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    x = np.zeros((n, d), np.float32)
    for i in range(n):
        x[i, 0] = 7.0 * rng.choice([-1, 1])
        for b0 in range(16, d, 16):
            blk = rng.choice(vals, size=16) * rng.choice([-1, 1], size=16)
            blk[rng.integers(16)] = 6.0 * rng.choice([-1, 1])
            x[i, b0:b0 + 16] = blk
    return x


def test_lossless_inputs_round_trip():
    rng = np.random.default_rng(3)
    x = _lossless_rows(rng, 6, 48)
    q = fp4_group_quant(x, 1)
    np.testing.assert_array_equal(q["scales"], np.float32(7.0 / 448.0))
    np.testing.assert_array_equal(q["scales"][:, None] * q["carrier"] / 6.0, x)


def test_single_key_closed_form():
    # Nk = 1: p = 1, y = 448, the key block's scale is 448 and P's code 6, so P's carrier is
    # 2688 = σ_P and O is exactly V's reconstruction g_c · 2688 / 6 = 448 g_c; V's entries are
    # 7 · 2^k, so g_c = |v_c| / 448 is exact and O is exactly v; with lossless Q and K rows
    # the LSE is exactly sm_scale · q·k (no smoothing: a single key's mean is the key)
    rng = np.random.default_rng(4)
    d = 48
    q = _lossless_rows(rng, 5, d)[None, None]
    k = _lossless_rows(rng, 1, d)[None, None]
    v = np.zeros((1, 1, 1, d), np.float32)
    v[0, 0, 0] = np.float32([7.0] + [0.0] * 15 + list(rng.choice([-7.0, 3.5, 0.875], 32)))
    r = sage_attention(q, k, v, sm_scale=0.01, gran=GRAN_PER_THREAD, smooth_k=False,
                       smooth_v=False, pv="fp4")
    np.testing.assert_array_equal(r["o"][0, 0], np.broadcast_to(v[0, 0, 0].astype(np.float64),
                                                               (5, d)))
    qk = q[0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64)
    np.testing.assert_allclose(r["lse"][0, 0], 0.01 * qk, rtol=1e-13, atol=1e-13)


def test_two_keys_closed_form():
    # head_dim 16, one query, two keys. q = (7, 3.5) and k = ((7, 0), (3.5, -7)) are lossless
    # (their group maximum 7 maps by 448/7 = 64 exactly onto 448, and the block codes are
    # (6, 3), (6, 0), (3, -6) at scale 448), so t = 0.05 q·k = (2.45, 0) exactly as rationals;
    # p2 = exp(-2.45); y = (448, fl32(448 p2)): the P block's scale is 448, ρ = fl32(6/448),
    # P's carriers are (2688, e2m1(fl32(y2 ρ)) · 448). V channel 0 = (7, -3.5) is lossless;
    # channel 1 = (1, 6) is worked through its first-level scale fl32(6/448) here.
    q = np.zeros((1, 1, 1, 16), np.float32); q[..., 0] = 7; q[..., 1] = 3.5
    k = np.zeros((1, 1, 2, 16), np.float32); k[0, 0, 0, 0] = 7; k[0, 0, 1, 0] = 3.5
    k[0, 0, 1, 1] = -7
    v = np.zeros((1, 1, 2, 16), np.float32); v[0, 0, 0, 0] = 7; v[0, 0, 1, 0] = -3.5
    v[0, 0, 0, 1] = 1; v[0, 0, 1, 1] = 6
    r = sage_attention(q, k, v, sm_scale=0.05, gran=GRAN_PER_THREAD, smooth_k=False,
                       smooth_v=False, pv="fp4")
    t1, t2 = 0.05 * 49.0, 0.0
    p2 = np.exp(t2 - t1)
    y2 = np.float32(448.0 * p2)
    rho = np.float32(np.float32(6.0) / np.float32(448.0))
    c2 = e2m1_decode(e2m1_encode(np.float32(y2 * rho)))
    r1 = np.float32(np.float32(448.0) / np.float32(6.0))
    u1 = (np.float32([1, 6]) * r1).astype(np.float32)
    s1 = e4m3_decode(e4m3_encode(np.abs(u1).max()))
    cv1 = e2m1_decode(e2m1_encode((u1 * np.float32(np.float32(6.0) / np.float32(s1))).astype(np.float32)))
    g1 = float(np.float32(np.float32(6.0) / np.float32(448.0)))
    vhat = np.array([[7.0, g1 * cv1[0] * s1 / 6.0], [-3.5, g1 * cv1[1] * s1 / 6.0]])
    pc = np.array([2688.0, c2 * 448.0])
    o = pc @ vhat / (2688.0 * (1.0 + p2))
    np.testing.assert_allclose(r["o"][0, 0, 0, :2], o, rtol=1e-13)
    np.testing.assert_allclose(r["lse"][0, 0, 0], t1 + np.log1p(p2), rtol=1e-13)
    assert c2 * 448.0 != 2688.0 * p2      # P's FP4 rounding is visible in the result


def test_p_quantisation_of_a_tile():
    # y = fl32(448 p) per 16 keys; the block holding the row maximum (p = 1) has scale 448
    p = np.exp(-np.linspace(0, 5, 40))[None, :]
    car = fp4_p(p)
    assert car[0, 0] == 2688.0
    assert np.all(car >= 0) and np.all(car <= 2688.0)
    y = (p * 448.0).astype(np.float32)
    assert np.all(np.abs(car / 6.0 - y) <= e4m3_decode(e4m3_encode(
        np.repeat([y[0, i:i + 16].max() for i in range(0, 40, 16)], 16)[:40])) / 6.0 + 1e-9)


@pytest.mark.parametrize("gran", [GRAN_PER_BLOCK, GRAN_PER_WARP, GRAN_PER_THREAD])
@pytest.mark.parametrize("causal", [False, True])
def test_fp4_bypass_equals_fp64(gran, causal):
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 2, 50, 40)).astype(np.float32)
    k = rng.standard_normal((1, 1, 70, 40)).astype(np.float32)
    v = rng.standard_normal((1, 1, 70, 40)).astype(np.float32)
    r = sage_attention(q, k, v, is_causal=causal, gran=gran, pv="fp4", bypass_quant=True,
                       smooth_k=True, smooth_v=True)
    kv = r["kv"][(0, 0)]
    for h in range(2):
        # exact over the float32-smoothed operands (the FP4 scale factors cancel exactly)
        of, lf = attention_fp64(q[0, h], kv["k_smoothed"], kv["v_smoothed"], r["sm_scale"], causal)
        of = of + kv["vbar"].astype(np.float64)
        lf = lf + r["sm_scale"] * (q[0, h].astype(np.float64) @ kv["kbar"].astype(np.float64))
        np.testing.assert_allclose(r["o"][0, h], of, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["lse"][0, h], lf, rtol=1e-12, atol=1e-12)


def test_fp4_close_to_fp64_and_coarser_than_fp8():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 2, 128, 64)).astype(np.float32)
    k = rng.standard_normal((1, 2, 300, 64)).astype(np.float32)
    v = rng.standard_normal((1, 2, 300, 64)).astype(np.float32)
    r4 = sage_attention(q, k, v, pv="fp4", accum=ACC_FP32)
    r8 = sage_attention(q, k, v, pv="fp8", accum=ACC_FP32)
    cos = lambda a, b: float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))
    for h in range(2):
        of, _ = attention_fp64(q[0, h], k[0, h], v[0, h], r4["sm_scale"], False)
        c4, c8 = cos(r4["o"][0, h], of), cos(r8["o"][0, h], of)
        assert 0.97 < c4 < c8


def test_fp4_online_single_tile_equals_final_form():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, 40, 32)).astype(np.float32)
    k = rng.standard_normal((1, 1, 100, 32)).astype(np.float32)
    v = rng.standard_normal((1, 1, 100, 32)).astype(np.float32)
    a = sage_attention(q, k, v, pv="fp4", p_max="final")
    b = sage_attention(q, k, v, pv="fp4", p_max="running")
    np.testing.assert_allclose(a["o"], b["o"], atol=1e-12)
    np.testing.assert_allclose(a["lse"], b["lse"], atol=1e-12)
