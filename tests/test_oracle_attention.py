"""Pins for the oracle's attention steps against exact mathematics.

- quantisation bypass (codes replaced by the values they encode) must equal float64
  softmax attention, O and LSE, for every mask/GQA/smoothing combination: this pins the
  score scaling, mask, softmax, normalisation, v̄ add-back and the LSE correction term;
- softmax invariance to smooth_k (q·k̄ is constant across keys);
- closed forms: Nk = 1, identical keys (uniform weights), constant V with smooth_v,
  causal row 0;
- head-dim zero padding is invisible;
- per-group scale indexing: groups of wildly different magnitude still give attention
  close to float64 (a wrong group index would not);
- scores are exact integers (brute-force Python loops);
- varlen == per-sequence dense.
"""

import numpy as np
import pytest

from oracle.attention import (ACC_FP16, ACC_FP16_FP32, ACC_FP32, attention_fp64,
                              attend_head, default_sm_scale, quantize_kv_head,
                              quantize_q_head, sage_attention, sage_attention_varlen, scores,
                              to_bf16, to_fp16)
from oracle.fp8 import e4m3_decode
from oracle.quant import GRAN_PER_BLOCK, GRAN_PER_THREAD, GRAN_PER_WARP

GRANS = [GRAN_PER_BLOCK, GRAN_PER_WARP, GRAN_PER_THREAD]


def _rand(shape, seed, scale=1.0, offset=0.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale + offset).astype(np.float16).astype(np.float32)


def _cos(a, b):
    a, b = np.ravel(a), np.ravel(b)
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("smooth_k,smooth_v", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("hq,hkv,nq,nk", [(2, 2, 40, 40), (4, 2, 33, 70), (3, 1, 70, 20)])
def test_bypass_equals_fp64_attention(causal, smooth_k, smooth_v, hq, hkv, nq, nk):
    d = 24
    q = _rand((1, hq, nq, d), 1)
    k = _rand((1, hkv, nk, d), 2, 1.0, 2.0)
    v = _rand((1, hkv, nk, d), 3, 1.0, -1.5)
    sm = 0.3
    res = sage_attention(q, k, v, is_causal=causal, sm_scale=sm, smooth_k=smooth_k,
                         smooth_v=smooth_v, bypass_quant=True)
    for h in range(hq):
        kv = res["kv"][(0, h // (hq // hkv))]
        # exact over the float32-smoothed operands: O = attn(q, K', V') + v̄ and
        # LSE = lse(q, K') + sm·q·k̄, to float64 rounding
        o, lse = attention_fp64(q[0, h], kv["k_smoothed"], kv["v_smoothed"], sm, causal)
        o = o + kv["vbar"].astype(np.float64)
        lse = lse + sm * (q[0, h].astype(np.float64) @ kv["kbar"].astype(np.float64))
        np.testing.assert_allclose(res["o"][0, h], o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(res["lse"][0, h], lse, rtol=1e-12, atol=1e-12)
        # and the unsmoothed definition, up to the float32 rounding of K - k̄, V - v̄
        o2, lse2 = attention_fp64(q[0, h], k[0, h // (hq // hkv)], v[0, h // (hq // hkv)], sm, causal)
        np.testing.assert_allclose(res["o"][0, h], o2, rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(res["lse"][0, h], lse2, rtol=1e-6, atol=1e-6)


def test_smooth_k_invariance_fp64():
    q = _rand((50, 16), 4)
    k = _rand((60, 16), 5, 1.0, 3.0)
    v = _rand((60, 16), 6)
    kbar = k.astype(np.float64).mean(axis=0)
    o1, l1 = attention_fp64(q, k, v, 0.25, False)
    o2, l2 = attention_fp64(q, k - kbar, v, 0.25, False)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l2 + 0.25 * (q.astype(np.float64) @ kbar), rtol=1e-12, atol=1e-12)


def test_causal_row_is_prefix_attention():
    q = _rand((1, 1, 30, 8), 7)
    k = _rand((1, 1, 30, 8), 8)
    v = _rand((1, 1, 30, 8), 9)
    res = sage_attention(q, k, v, is_causal=True, sm_scale=0.5, smooth_k=False, bypass_quant=True)
    for i in (0, 5, 29):
        o, _ = attention_fp64(q[0, 0, i:i + 1], k[0, 0, :i + 1], v[0, 0, :i + 1], 0.5, False)
        np.testing.assert_allclose(res["o"][0, 0, i], o[0], rtol=1e-12)


@pytest.mark.parametrize("accum", [ACC_FP32, ACC_FP16_FP32])
@pytest.mark.parametrize("smooth_v", [False, True])
def test_single_key_gives_dequantised_v0(accum, smooth_v):
    q = _rand((1, 2, 20, 16), 10)
    k = _rand((1, 2, 1, 16), 11)
    v = _rand((1, 2, 1, 16), 12, 3.0, 1.0)
    res = sage_attention(q, k, v, accum=accum, smooth_v=smooth_v, gran=GRAN_PER_THREAD)
    for h in range(2):
        kv = res["kv"][(0, h)]
        expect = e4m3_decode(kv["v8"][0]) * kv["sv"].astype(np.float64) + kv["vbar"]
        np.testing.assert_allclose(res["o"][0, h], np.broadcast_to(expect, (20, 16)), rtol=1e-12, atol=1e-12)


def test_identical_keys_give_uniform_weights():
    q = _rand((1, 1, 17, 32), 13)
    k = np.broadcast_to(_rand((1, 1, 1, 32), 14), (1, 1, 200, 32)).copy()
    v = _rand((1, 1, 200, 32), 15)
    res = sage_attention(q, k, v, accum=ACC_FP32, smooth_k=True)
    kv = res["kv"][(0, 0)]
    assert np.all(kv["k8"] == 0)                 # K - mean(K) = 0 exactly
    expect = e4m3_decode(kv["v8"]).mean(axis=0) * kv["sv"]
    np.testing.assert_allclose(res["o"][0, 0], np.broadcast_to(expect, (17, 32)), rtol=1e-12, atol=1e-12)
    res16 = sage_attention(q, k, v, accum=ACC_FP16_FP32, smooth_k=True)
    np.testing.assert_allclose(res16["o"][0, 0], np.broadcast_to(expect, (17, 32)), rtol=1e-12, atol=1e-12)


def test_constant_v_with_smooth_v_gives_mean():
    q = _rand((1, 1, 10, 8), 16)
    k = _rand((1, 1, 50, 8), 17)
    v = np.broadcast_to(np.float32([1.5, -2.0, 0.0, 7.25, 3.0, -0.5, 0.125, 10.0]), (1, 1, 50, 8)).copy()
    res = sage_attention(q, k, v, smooth_v=True)
    assert np.all(res["kv"][(0, 0)]["sv"] == 0)
    np.testing.assert_array_equal(res["o"][0, 0], np.broadcast_to(v[0, 0, 0].astype(np.float64), (10, 8)))


def test_causal_row_zero_sees_only_key_zero():
    q = _rand((1, 1, 64, 16), 18)
    k = _rand((1, 1, 64, 16), 19)
    v = _rand((1, 1, 64, 16), 20)
    res = sage_attention(q, k, v, is_causal=True, smooth_v=True)
    kv = res["kv"][(0, 0)]
    expect = e4m3_decode(kv["v8"][0]) * kv["sv"] + kv["vbar"]
    np.testing.assert_allclose(res["o"][0, 0, 0], expect, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("gran", GRANS)
def test_head_dim_zero_padding_is_invisible(gran):
    d, dp = 72, 128
    q = _rand((1, 2, 90, d), 21)
    k = _rand((1, 2, 90, d), 22, 1.0, 1.0)
    v = _rand((1, 2, 90, d), 23)
    pad = lambda t: np.concatenate([t, np.zeros(t.shape[:-1] + (dp - d,), np.float32)], -1)
    sm = default_sm_scale(d)
    a = sage_attention(q, k, v, sm_scale=sm, gran=gran, smooth_v=True)
    b = sage_attention(pad(q), pad(k), pad(v), sm_scale=sm, gran=gran, smooth_v=True)
    np.testing.assert_array_equal(a["o"], b["o"][..., :d])
    np.testing.assert_array_equal(a["lse"], b["lse"])
    assert np.all(b["o"][..., d:] == 0)


@pytest.mark.parametrize("gran", GRANS)
def test_group_scales_are_indexed_per_group(gran):
    # every 16-token K group and every Q row has its own magnitude (factors up to 2^6);
    # attention on such data stays close to fp64 only if each score uses its own group's
    # scales (a shifted or transposed index would mix magnitudes of 64x)
    n, d = 256, 32
    q = _rand((1, 1, n, d), 24) * (2.0 ** (np.arange(n) % 7))[None, None, :, None].astype(np.float32)
    k = _rand((1, 1, n, d), 25) * (2.0 ** -((np.arange(n) // 16) % 7))[None, None, :, None].astype(np.float32)
    v = _rand((1, 1, n, d), 26)
    sm = 0.02
    res = sage_attention(q, k, v, sm_scale=sm, gran=gran)
    o, _ = attention_fp64(q[0, 0], k[0, 0], v[0, 0], sm, False)
    assert _cos(res["o"][0, 0], o) > 0.99


@pytest.mark.parametrize("accum", [ACC_FP32, ACC_FP16_FP32])
def test_quantised_close_to_fp64_on_tiny_workload(accum):
    q = _rand((1, 2, 256, 64), 27)
    k = _rand((1, 2, 256, 64), 28)
    v = _rand((1, 2, 256, 64), 29)
    sm = default_sm_scale(64)
    res = sage_attention(q, k, v, sm_scale=sm, gran=GRAN_PER_BLOCK, accum=accum)
    for h in range(2):
        o, lse = attention_fp64(q[0, h], k[0, h], v[0, h], sm, False)
        assert _cos(res["o"][0, h], o) > 0.99
        assert np.abs(res["lse"][0, h] - lse).max() < 0.05


def test_scores_are_exact_integers():
    rng = np.random.default_rng(30)
    q8 = rng.integers(-127, 128, (5, 9)).astype(np.int8)
    k8 = rng.integers(-127, 128, (7, 9)).astype(np.int8)
    s = scores(q8, k8)
    for i in range(5):
        for j in range(7):
            assert s[i, j] == sum(int(q8[i, c]) * int(k8[j, c]) for c in range(9))
    ext = np.full((1, 128), 127, np.int8)
    assert scores(ext, -ext)[0, 0] == -128 * 127 * 127


def test_varlen_equals_per_sequence_dense():
    lens = [5, 130, 1, 64]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    t = int(cu[-1])
    q = _rand((t, 4, 16), 31)
    k = _rand((t, 2, 16), 32, 1.0, 1.0)
    v = _rand((t, 2, 16), 33)
    res = sage_attention_varlen(q, k, v, cu, cu, is_causal=True, smooth_v=True, sm_scale=0.25)
    for b, n in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        d = sage_attention(q[sl].transpose(1, 0, 2)[None], k[sl].transpose(1, 0, 2)[None],
                           v[sl].transpose(1, 0, 2)[None], is_causal=True, smooth_v=True, sm_scale=0.25)
        np.testing.assert_array_equal(res["o"][sl], d["o"][0].transpose(1, 0, 2))
        np.testing.assert_array_equal(res["lse"][:, sl], d["lse"][0])


def test_rows_subset_matches_full():
    q = _rand((1, 1, 300, 32), 34)
    k = _rand((1, 1, 200, 32), 35)
    v = _rand((1, 1, 200, 32), 36)
    full = sage_attention(q, k, v, gran=GRAN_PER_WARP)
    rows = np.array([0, 31, 32, 299])
    part = sage_attention(q, k, v, gran=GRAN_PER_WARP, rows=rows)
    np.testing.assert_array_equal(part["o"][0, 0], full["o"][0, 0, rows])


def test_argument_errors():
    q = _rand((1, 3, 4, 8), 37)
    k = _rand((1, 2, 4, 8), 38)
    with pytest.raises(ValueError):
        sage_attention(q, k, k)
    with pytest.raises(NotImplementedError):
        sage_attention(q[:, :2], k, k, accum=ACC_FP16)
    with pytest.raises(ValueError):
        sage_attention(_rand((1, 1, 4, 130), 1), _rand((1, 1, 4, 130), 2), _rand((1, 1, 4, 130), 3))


def test_output_rounding_helpers():
    assert to_fp16(np.float64(1.0 + 2.0**-11)) == 1.0        # tie -> even
    assert to_fp16(np.float64(1.0 + 3 * 2.0**-11)) == 1.0 + 2.0**-9
    assert to_fp16(np.float64(65520.0)) == np.inf             # rounds past max
    assert to_fp16(np.float64(2.0**-25)) == 0.0               # half the smallest subnormal
    assert to_bf16(np.float64(1.0 + 2.0**-8)) == 1.0
    assert to_bf16(np.float64(1.0 + 3 * 2.0**-8)) == 1.0 + 2.0**-6
    x = np.random.default_rng(39).standard_normal(1000)
    np.testing.assert_array_equal(to_fp16(x), x.astype(np.float16).astype(np.float64))


def _e4m3_nearest(x):
    """Round a positive real to the E4M3 grid by scanning the stored value table (nearest,
    ties to the even code), independently of the oracle's encoder."""
    import os
    from fractions import Fraction
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "e4m3_positive_values.txt")
    vals = []
    with open(path) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                c, v = ln.split()
                vals.append((float(Fraction(v)), int(c, 16)))
    best = min(vals, key=lambda t: (abs(t[0] - x), t[1] & 1))
    return best[0]


@pytest.mark.parametrize("accum", [ACC_FP32, ACC_FP16_FP32])
def test_two_keys_closed_form(accum):
    # head_dim 1, one query, two keys: every quantisation step can be done by hand.
    #   q = 1 -> code 127, s_q = fl32(1/127);  k = (1, 0.5) -> one K group, codes (127, 64)
    #   (0.5 * fl32(127) = 63.5 rounds to even 64), s_k = fl32(1/127); scores 16129 and 8128;
    #   v = (2, -1) -> s_v = fl32(2/448), codes 448 and -224 (both exact in E4M3).
    # With sm_scale = 10: t_j = S_j s_q s_k 10, p2 = exp(t2 - t1) ~ 0.0070; every accumulation
    # mode scales P by 448 before its E4M3 rounding: P~ = (448, e4m3(448 p2)), l = 1 + p2
    # (unquantised), O = (P~1 V~1 + P~2 V~2) s_v / (448 l), LSE = t1 + ln l.
    q = np.float32([[[[1.0]]]])
    k = np.float32([[[[1.0], [0.5]]]])
    v = np.float32([[[[2.0], [-1.0]]]])
    res = sage_attention(q, k, v, sm_scale=10.0, gran=GRAN_PER_THREAD, accum=accum, smooth_k=False)
    kv, qq = res["kv"][(0, 0)], res["q"][(0, 0)]
    assert qq["q8"].ravel().tolist() == [127] and kv["k8"].ravel().tolist() == [127, 64]
    s_qk = float(np.float32(1.0) / np.float32(127.0))
    s_v = float(np.float32(2.0) / np.float32(448.0))
    t1, t2 = 16129.0 * s_qk * s_qk * 10.0, 8128.0 * s_qk * s_qk * 10.0
    p2 = np.exp(t2 - t1)
    pt2 = _e4m3_nearest(448.0 * p2)
    assert pt2 != _e4m3_nearest(p2) * 448.0          # the scale of P is visible here
    l = 1.0 + p2
    o = (448.0 * 448.0 + pt2 * -224.0) * s_v / (448.0 * l)
    np.testing.assert_allclose(res["o"][0, 0, 0, 0], o, rtol=1e-14)
    np.testing.assert_allclose(res["lse"][0, 0, 0], t1 + np.log(l), rtol=1e-14)
