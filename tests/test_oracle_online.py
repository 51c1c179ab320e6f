"""The oracle's online form (p_max="running": P~ quantised against the running maximum of the
128-key tiles seen so far, accumulator and row sum rescaled by exp(m_old - m_new)), pinned
against the final-max form and against exact attention:
- one key tile: both forms take the same maximum, so every output bit agrees;
- codes bypassed (P unrounded, scales 1): the rescaling algebra must give exact attention,
  causal or not (a dropped or wrong rescale factor fails here);
- every row's maximum in its first tile (the maximum never moves): same P~ as the final form,
  so the outputs agree up to float64 summation order, in every accumulation mode;
- in general the two forms differ only by E4M3 rounding of P~ (cosine close to 1)."""

import numpy as np
import pytest

from oracle.attention import (ACC_FP16_FP32, ACC_FP32, GRAN_PER_THREAD, GRAN_PER_WARP,
                              attention_fp64, sage_attention)
from oracle.quant import K_GROUP, Q_GROUP


def _rand(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


@pytest.mark.parametrize("key_tile", [96, 128])
def test_single_tile_forms_identical(key_tile):
    nk = key_tile
    q, k, v = _rand((1, 2, 90, 64), 1), _rand((1, 2, nk, 64), 2), _rand((1, 2, nk, 64), 3)
    for accum in (ACC_FP32, ACC_FP16_FP32):
        a = sage_attention(q, k, v, accum=accum, p_max="final")
        b = sage_attention(q, k, v, accum=accum, p_max="running", key_tile=key_tile)
        np.testing.assert_array_equal(a["o"], b["o"])
        np.testing.assert_array_equal(a["lse"], b["lse"])


@pytest.mark.parametrize("key_tile", [96, 128, 7])
@pytest.mark.parametrize("causal", [False, True])
def test_bypassed_codes_give_exact_attention(causal, key_tile):
    q, k, v = _rand((1, 1, 200, 32), 4), _rand((1, 1, 333, 32), 5), _rand((1, 1, 333, 32), 6)
    r = sage_attention(q, k, v, is_causal=causal, bypass_quant=True, p_max="running",
                       smooth_k=False, key_tile=key_tile)
    o, lse = attention_fp64(q[0, 0], k[0, 0], v[0, 0], r["sm_scale"], causal)
    np.testing.assert_allclose(r["o"][0, 0], o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["lse"][0, 0], lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("key_tile", [96, 128])
@pytest.mark.parametrize("accum", [ACC_FP32, ACC_FP16_FP32])
def test_maximum_in_first_tile_matches_final_form(accum, key_tile):
    # positive queries and a positive first key: key 0 has every row's largest score (by ~7
    # natural-log units), while the other keys keep non-zero E4M3 probabilities
    q = np.abs(_rand((1, 2, 64, 64), 7)) + 0.1
    k = _rand((1, 2, 400, 64), 8)
    k[:, :, 0, :] = 1.5
    v = _rand((1, 2, 400, 64), 9)
    a = sage_attention(q, k, v, accum=accum, gran=GRAN_PER_THREAD, smooth_k=False, p_max="final")
    b = sage_attention(q, k, v, accum=accum, gran=GRAN_PER_THREAD, smooth_k=False, p_max="running",
                       key_tile=key_tile)
    for h in range(2):                                 # the premise: key 0 is every row's max
        kq, qq = a["kv"][(0, h)], a["q"][(0, h)]
        t = (qq["q8"].astype(np.float64) @ kq["k8"].astype(np.float64).T
             * qq["sq"].astype(np.float64)[np.arange(64) // Q_GROUP[GRAN_PER_THREAD]][:, None]
             * kq["sk"].astype(np.float64)[np.arange(400) // K_GROUP[GRAN_PER_THREAD]][None, :])
        assert (np.argmax(t, axis=1) == 0).all()
    np.testing.assert_allclose(b["o"], a["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=0, atol=1e-12)


def test_forms_differ_only_by_p_rounding():
    q, k, v = _rand((1, 2, 256, 128), 10), _rand((1, 2, 1024, 128), 11), _rand((1, 2, 1024, 128), 12)
    a = sage_attention(q, k, v, gran=GRAN_PER_WARP, p_max="final")
    b = sage_attention(q, k, v, gran=GRAN_PER_WARP, p_max="running")
    assert not np.array_equal(a["o"], b["o"])
    x, y = a["o"].ravel(), b["o"].ravel()
    assert x @ y / np.linalg.norm(x) / np.linalg.norm(y) > 0.999
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=0, atol=1e-9)


def test_rejects_unknown_form():
    q = _rand((1, 1, 4, 8), 13)
    with pytest.raises(ValueError):
        sage_attention(q, q, q, p_max="lagging")


def test_fp16_pv_variant_online_form():
    # pv="fp16": one key tile gives the final form's bits; bypassed codes give exact attention
    q, k, v = _rand((1, 2, 70, 64), 14), _rand((1, 2, 120, 64), 15), _rand((1, 2, 120, 64), 16)
    a = sage_attention(q, k, v, pv="fp16", p_max="final")
    b = sage_attention(q, k, v, pv="fp16", p_max="running")
    np.testing.assert_array_equal(a["o"], b["o"])
    q, k, v = _rand((1, 1, 150, 32), 17), _rand((1, 1, 300, 32), 18), _rand((1, 1, 300, 32), 19)
    r = sage_attention(q, k, v, is_causal=True, bypass_quant=True, pv="fp16", p_max="running",
                       smooth_k=False)
    o, _ = attention_fp64(q[0, 0], k[0, 0], v[0, 0], r["sm_scale"], True)
    np.testing.assert_allclose(r["o"][0, 0], o, rtol=0, atol=1e-12)


def test_varlen_online_form_equals_per_sequence_dense():
    from oracle.attention import sage_attention_varlen
    rng = np.random.default_rng(20)
    lens = [150, 1, 300]
    t = sum(lens)
    q = rng.standard_normal((t, 4, 32)).astype(np.float32)
    k = rng.standard_normal((t, 2, 32)).astype(np.float32)
    v = rng.standard_normal((t, 2, 32)).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    res = sage_attention_varlen(q, k, v, cu, cu, is_causal=True, p_max="running")
    for b in range(3):
        sl = slice(cu[b], cu[b + 1])
        d = sage_attention(q[sl].transpose(1, 0, 2)[None], k[sl].transpose(1, 0, 2)[None],
                           v[sl].transpose(1, 0, 2)[None], is_causal=True, p_max="running")
        np.testing.assert_array_equal(res["o"][sl], d["o"][0].transpose(1, 0, 2))
        np.testing.assert_array_equal(res["lse"][:, sl], d["lse"][0])
