"""Degenerate inputs, against the oracle: every quantisation group at absmax 0 (all-zero
tensors), keys constant over the sequence (smooth_k leaves K' = 0, so every score is 0 and
attention is a plain mean of V), values constant over the sequence (smooth_v leaves V' = 0 and
the V scale 0, so the output is the constant itself), and Q near the fp16 maximum with K among
the fp16 subnormals. (Scores far beyond fp32's resolution, e.g. both Q and K in the thousands,
are outside the method: its softmax runs in fp32, so the oracle's fp64 ranking of near-equal
maxima cannot be reproduced there.)
Bit-exact where the codes, scales and scores are compared; the output within the usual
tolerance, or exact where the mathematics makes it exact. Every case runs on both
implementations of a dense call (the main pipeline and the one-launch short-sequence
kernel)."""

import numpy as np
import pytest
import torch

from oracle.attention import sage_attention
from quantized_attention_mean_gb300.workloads import Workload, dense_inputs, to_hnd_f32

from helpers import (TOL_COS, TOL_LSE, TOL_MAX_ABS, cosine, max_abs_excess, oracle_kw, out_to_hnd, run_gpu_dense,
                     short_eligible)

pytestmark = pytest.mark.gpu


PATHS = ["main", "short"]


def _check(w, q, k, v, exact_out=False, path="main"):
    import quantized_attention_mean_gb300 as qa
    if path == "short" and not short_eligible(w):
        pytest.skip("too long for the short-sequence kernel")
    g = run_gpu_dense(w, q, k, v, debug_scores=path == "main", path=path)
    assert g["status"] == 0
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    ref = sage_attention(qn, kn, vn, **oracle_kw(w))
    ex = {n: t.cpu().numpy() for n, t in qa.export_quant(g["ws"], w.B, w.Hq, w.Hkv, w.Nq, w.Nk,
                                                          w.d, w.gran).items()}
    for b in range(w.B):
        for h in range(w.Hq):
            np.testing.assert_array_equal(ex["q8"][b, h], ref["q"][(b, h)]["q8"])
            np.testing.assert_array_equal(ex["sq"][b, h].view(np.uint32), ref["q"][(b, h)]["sq"].view(np.uint32))
        for h in range(w.Hkv):
            kv = ref["kv"][(b, h)]
            np.testing.assert_array_equal(ex["k8"][b, h], kv["k8"])
            np.testing.assert_array_equal(ex["sk"][b, h].view(np.uint32), kv["sk"].view(np.uint32))
            np.testing.assert_array_equal(ex["v8"][b, h], kv["v8"])
            np.testing.assert_array_equal(ex["vscale"][b, h].view(np.uint32), kv["sv"].view(np.uint32))
    o = out_to_hnd(g["out"], w.layout)
    assert np.isfinite(o).all()
    if exact_out:
        np.testing.assert_array_equal(o, ref["o"].astype(np.float16).astype(np.float32))
    assert max_abs_excess(o, ref["o"], w.dtype) <= TOL_MAX_ABS
    if np.abs(ref["o"]).max() > 0:
        assert cosine(o, ref["o"]) >= TOL_COS
    if w.return_lse:
        assert np.abs(g["lse"].cpu().numpy() - ref["lse"]).max() <= TOL_LSE
    return o, g, ref


@pytest.mark.parametrize("path", PATHS)
def test_all_zero_inputs(path):
    w = Workload("zeros", 1, 2, 2, 200, 250, 64, gran="per_warp", return_lse=True, smooth_v=True)
    q, k, v = (torch.zeros_like(t) for t in dense_inputs(w, 0))
    o, g, ref = _check(w, q, k, v, exact_out=True, path=path)
    assert not o.any()
    # every score 0: the LSE is ln(Nk) exactly up to the log's rounding
    np.testing.assert_allclose(g["lse"].cpu().numpy(), np.log(w.Nk), atol=1e-5)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("causal", [False, True])
def test_keys_constant_over_tokens(causal, path):
    w = Workload("const_k", 2, 4, 2, 250, 250, 128, dtype="bf16", layout="NHD", is_causal=causal,
                 gran="per_thread", accum="fp32", return_lse=True)
    q, k, v = dense_inputs(w, 1)
    k = k[:, :1].expand_as(k).contiguous()          # NHD: the first token's keys everywhere
    o, g, ref = _check(w, q, k, v, path=path)
    if path == "main":
        assert not g["scores"].cpu().numpy()[g["scores"].cpu().numpy() != -2**31].any()
    # uniform attention: the (causal) running mean of V, up to V's E4M3 rounding (rows that
    # average at least 32 keys)
    vn = to_hnd_f32(v, w.layout).astype(np.float64)
    grp = w.Hq // w.Hkv
    for h in range(w.Hq):
        vh = vn[0, h // grp]
        mean = np.cumsum(vh, 0) / np.arange(1, w.Nk + 1)[:, None] if causal else np.broadcast_to(vh.mean(0), vh.shape)
        assert np.abs(o[0, h, 31:] - mean[31:]).max() < 0.05


@pytest.mark.parametrize("path", PATHS)
def test_values_constant_over_tokens(path):
    w = Workload("const_v", 1, 2, 1, 150, 233, 64, gran="per_block", accum="fp16+fp32", smooth_v=True,
                 return_lse=True)
    q, k, v = dense_inputs(w, 2)
    v = v[:, :, :1].expand_as(v).contiguous()       # HND: the first token's values everywhere
    o, g, ref = _check(w, q, k, v, path=path)
    # V' = 0 and s_v = 0: the output is v-mean, i.e. the constant row, in every query row
    vrow = v[0, 0, 0].float().numpy()
    assert np.array_equal(o[0, 0], np.broadcast_to(vrow, o[0, 0].shape))
    assert np.array_equal(o[0, 1], np.broadcast_to(vrow, o[0, 1].shape))


@pytest.mark.parametrize("path", PATHS)
def test_inputs_at_the_fp16_extremes(path):
    # Q near the fp16 maximum, K down among fp16 subnormals (their products, and so the
    # softmax, stay ordinary): the scales and the fixed-point K mean at both ends of the range
    w = Workload("extremes", 1, 2, 2, 256, 256, 64, gran="per_thread", accum="fp32", return_lse=True,
                 smooth_v=True)
    q, k, v = dense_inputs(w, 3)
    q = (q.float() * 1.5e4).clamp(-6.5e4, 6.5e4).half()
    k = (k.float() * 4e-5).half()
    assert (k.abs() < 6.1e-5).float().mean() > 0.5  # mostly subnormal
    _check(w, q, k, v, path=path)


@pytest.mark.parametrize("heads,n", [(2, 1000), (128, 4096)], ids=["one_batch_per_block", "four_batches_per_block"])
def test_bf16_means_beyond_the_packed_sum(heads, n):
    # bf16 K and V with nonzero magnitudes below 2^-17 in some rows of some heads and
    # magnitudes of 2^14 and more in others (a third of the heads stays ordinary): the
    # statistics pass's packed fixed-point sum covers neither, so those warps redo their rows
    # with exact int64 conversions; every smoothing mean stays bit-exact. The larger case
    # gives each statistics block four batches of rows.
    import quantized_attention_mean_gb300 as qa
    from oracle.quant import fixed_point_mean
    w = Workload("bf16_ranges", 1, heads, heads, 128, n, 64, dtype="bf16", gran="per_warp",
                 accum="fp16+fp32", smooth_v=True)
    q, k, v = dense_inputs(w, 5)
    k, v = k.float(), v.float()
    k[:, 0::3, 3::97, :] *= 2.0 ** -20          # |x| ~ 1e-6, below 2^-17 = 7.6e-6
    v[:, 0::3, 11::83, :] *= 2.0 ** -21
    k[:, 1::3, 5::89, 7] = 3.0e4                # above the packed sum's 2^14
    v[:, 1::3, 17::101, 3] = -2.5e4
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    g = run_gpu_dense(w, q, k, v, path="main")
    assert g["status"] == 0
    ex = qa.export_quant(g["ws"], w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran)
    km, vm = ex["kmean"].cpu().numpy(), ex["vmean"].cpu().numpy()
    kn, vn = to_hnd_f32(k, w.layout), to_hnd_f32(v, w.layout)
    for h in range(heads):
        np.testing.assert_array_equal(km[0, h].view(np.uint32), fixed_point_mean(kn[0, h]).view(np.uint32))
        np.testing.assert_array_equal(vm[0, h].view(np.uint32), fixed_point_mean(vn[0, h]).view(np.uint32))
