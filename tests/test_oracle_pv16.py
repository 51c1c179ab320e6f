"""Pins for the oracle's FP16 P·V variant (INT8 Q/K, fp16 P and V')."""

import numpy as np
import pytest

from oracle.attention import (ACC_FP16_FP32, ACC_FP32, attend_head, attention_fp64,
                              quantize_kv_head, sage_attention, to_fp16)
from oracle.quant import GRAN_PER_THREAD, GRAN_PER_WARP


def _rand(seed, nq, nk, d, scale=1.0):
    rng = np.random.default_rng(seed)
    f = lambda *s: (rng.normal(size=s) * scale).astype(np.float32)
    return f(nq, d), f(nk, d), f(nk, d)


def test_single_key_gives_the_fp16_value():
    # one key: p = 1 exactly, so O = fp16(V) row for every query
    q, k, v = _rand(1, 9, 1, 24)
    kvq = quantize_kv_head(k, v, GRAN_PER_WARP, smooth_k=True, smooth_v=False, pv="fp16")
    o = attend_head(q, kvq, gran=GRAN_PER_WARP, sm_scale=0.2, is_causal=False, accum=ACC_FP32)["o"]
    np.testing.assert_array_equal(o, np.broadcast_to(to_fp16(v[0].astype(np.float64)), o.shape))


def test_constant_v_with_smoothing_is_exact():
    q, k, _ = _rand(2, 17, 40, 32)
    v = np.tile(np.linspace(-3, 5, 32, dtype=np.float32), (40, 1))
    kvq = quantize_kv_head(k, v, GRAN_PER_WARP, True, True, pv="fp16")
    o = attend_head(q, kvq, gran=GRAN_PER_WARP, sm_scale=0.3, is_causal=True, accum=ACC_FP32)["o"]
    np.testing.assert_array_equal(o, np.broadcast_to(kvq["vbar"].astype(np.float64), o.shape))


@pytest.mark.parametrize("accum", [ACC_FP32, ACC_FP16_FP32])
def test_pv_rounding_within_fp16_bound(accum):
    # Q/K codes bypassed: what remains is fp16 rounding of P (values <= 1) and of V'; each is
    # a relative error <= 2^-11 (plus 2^-25 absolute for subnormal P) in every
    # accumulation mode
    q, k, v = _rand(3, 33, 300, 64, scale=1.3)
    kvq = quantize_kv_head(k, v, GRAN_PER_THREAD, True, True, pv="fp16")
    o = attend_head(q, kvq, gran=GRAN_PER_THREAD, sm_scale=0.125, is_causal=False, accum=accum,
                    bypass_quant="qk")["o"]
    o_exact, _ = attention_fp64(q, kvq["k_smoothed"], kvq["v_smoothed"], 0.125, False)
    o_exact = o_exact + kvq["vbar"].astype(np.float64)
    vmax = float(np.abs(kvq["v_smoothed"]).max())
    bound = 2.0 ** -10 * 1.01 * vmax + 300 * 2.0 ** -25 * vmax
    assert np.max(np.abs(o - o_exact)) <= bound


def test_fp16_pv_is_closer_to_exact_than_fp8():
    rng = np.random.default_rng(4)
    q = rng.normal(size=(1, 2, 128, 64)).astype(np.float32)
    k = rng.normal(size=(1, 2, 256, 64)).astype(np.float32)
    v = rng.normal(size=(1, 2, 256, 64)).astype(np.float32)
    r16 = sage_attention(q, k, v, pv="fp16")
    r8 = sage_attention(q, k, v, pv="fp8")
    err = lambda o: max(np.max(np.abs(o[0, h] - attention_fp64(q[0, h], k[0, h], v[0, h],
                                                                r16["sm_scale"], False)[0]))
                        for h in range(2))
    assert err(r16["o"]) < err(r8["o"])


def test_rejects_unknown_pv():
    q, k, v = _rand(5, 4, 4, 8)
    with pytest.raises(ValueError):
        quantize_kv_head(k, v, GRAN_PER_WARP, True, False, pv="int4")
