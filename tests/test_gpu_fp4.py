"""GPU parity of the FP4 microscaled variant (sage_attn_fp4) against the oracle's pv="fp4"
emulation, through the C ABI.

Bit-exact: the E2M1 converter, the fp16 carriers (E2M1 code x E4M3 block scale) of Q, K and
V', the first-level scales s_q / s_k / s_v and the smoothing means.
Tolerance, derived from the oracle itself (tests/test_oracle_fp4.py and a CPU study of the
same cases): against the oracle's online form (the kernel's form) a relative perturbation of
1e-7 in the scores, the size of the GPU's ex2.approx and fp32 summation differences, flips
an E2M1 rounding of P now and then, which moves a few outputs by up to 3e-3 (at most 6e-4 of
them beyond 1e-3) at cosine 0.9999999: the bounds are max-abs 2e-2 beyond half an output ulp,
at most 0.2% of elements beyond 1e-3, cosine >= 0.99999 and LSE within 1e-4. Against the
final form the oracle's own two forms differ by up to 3.5e-2 (cosine >= 0.9993): max-abs 5e-2
and cosine >= 0.999. Against fp64 attention FP4 itself reaches cosine ~0.98 on these inputs:
>= 0.97.
"""

import numpy as np
import pytest
import torch

from helpers import cosine, excess_fraction, gpu_kw, max_abs_excess, oracle_kw, out_to_hnd
from oracle.attention import attention_fp64, sage_attention
from oracle.fp4 import e2m1_encode
from quantized_attention_mean_gb300.workloads import WORKLOADS, Workload, dense_inputs, to_hnd_f32

pytestmark = pytest.mark.gpu

TOL4_ONLINE_MAX_ABS = 2e-2
TOL4_ONLINE_ELEM = 1e-3
TOL4_ONLINE_ELEM_FRAC = 2e-3
TOL4_ONLINE_COS = 0.99999
TOL4_ONLINE_LSE = 1e-4
TOL4_FINAL_MAX_ABS = 5e-2
TOL4_FINAL_COS = 0.999
TOL4_COS_FP64 = 0.97
TOL4_LSE = 2e-2

CASES = [
    WORKLOADS["tiny"],
    Workload("ragged_fp16", 1, 2, 2, 300, 300, 64, gran="per_warp", accum="fp32"),
    Workload("gqa_nhd_bf16", 2, 4, 2, 200, 333, 128, dtype="bf16", layout="NHD", gran="per_thread",
             accum="fp32", return_lse=True, k_offset_std=3.0),
    Workload("causal_gqa", 1, 8, 2, 384, 384, 128, dtype="bf16", layout="NHD", is_causal=True,
             gran="per_thread", accum="fp32", return_lse=True, k_offset_std=3.0),
    Workload("causal_ragged", 2, 2, 2, 270, 270, 64, is_causal=True, gran="per_block", return_lse=True),
    Workload("dit_like", 1, 3, 3, 500, 500, 64, dtype="bf16", gran="per_warp", accum="fp16+fp32",
             smooth_v=True, k_offset_std=4.0, v_offset_std=2.0, return_lse=True),
    Workload("d128_512", 1, 2, 2, 512, 512, 128, gran="per_warp", accum="fp32", return_lse=True),
    Workload("pad_d72", 1, 2, 1, 140, 260, 72, dtype="bf16", gran="per_thread", accum="fp32+fp32"),
    Workload("pad_d40_nhd", 1, 2, 2, 160, 200, 40, layout="NHD", gran="per_block", smooth_v=True,
             v_offset_std=1.0),
    Workload("short_keys", 1, 2, 2, 129, 1, 64, gran="per_warp", smooth_v=True),
    Workload("one_tile_long_keys", 1, 2, 2, 100, 1000, 64, gran="per_warp", return_lse=True),
]

_cache = {}


def _run(w):
    if w.name in _cache:
        return _cache[w.name]
    import quantized_attention_mean_gb300 as qa
    q, k, v = dense_inputs(w, 0)
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    dev = torch.device("cuda:0")
    ws = qa.alloc_workspace(qa.workspace_bytes(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran), dev)
    res = qa.sage_attn_fp4(q.to(dev), k.to(dev), v.to(dev), workspace=ws, **gpu_kw(w))
    out, lse = res if w.return_lse else (res, None)
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    ex = {n: t.cpu().numpy() for n, t in qa.export_quant(ws, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d,
                                                          w.gran).items()}
    ex16 = {n: t.cpu().numpy() for n, t in qa.export_fp16(ws, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d,
                                                           w.gran).items()}
    g = dict(o=out_to_hnd(out, w.layout), lse=None if lse is None else lse.cpu().numpy(),
             ex=ex, ex16=ex16, qn=qn, kn=kn, vn=vn)
    _cache.clear()
    _cache[w.name] = g
    return g


def test_e2m1_conversion_matches_oracle():
    import quantized_attention_mean_gb300 as qa
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(1 << 18).astype(np.float32) * s for s in (0.1, 1, 3, 10)]
    grid = np.arange(-8.0, 8.0, 1.0 / 256.0, dtype=np.float32)
    ties = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 1e30, 0.0])
    near = np.concatenate([np.nextafter(ties, np.float32(-1e38)), np.nextafter(ties, np.float32(1e38))])
    x = np.concatenate(vals + [grid, ties, near])
    x = np.concatenate([x, -x])
    got = qa.e2m1(torch.from_numpy(x).cuda()).cpu().numpy()
    np.testing.assert_array_equal(got, e2m1_encode(x))


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_fp4_quantisation_bit_exact(w):
    g = _run(w)
    ref = sage_attention(g["qn"], g["kn"], g["vn"], pv="fp4", **oracle_kw(w), rows=[0])
    ex, ex16 = g["ex"], g["ex16"]
    for b in range(w.B):
        for h in range(w.Hq):
            qq = ref["q"][(b, h)]
            np.testing.assert_array_equal(ex16["q16"][b, h].astype(np.float64), qq["q4"])
            np.testing.assert_array_equal(ex["sq"][b, h].view(np.uint32), qq["sq"].view(np.uint32))
        for h in range(w.Hkv):
            kv = ref["kv"][(b, h)]
            np.testing.assert_array_equal(ex["kmean"][b, h].view(np.uint32), kv["kbar"].view(np.uint32))
            np.testing.assert_array_equal(ex16["k16"][b, h].astype(np.float64), kv["k4"])
            np.testing.assert_array_equal(ex["sk"][b, h].view(np.uint32), kv["sk"].view(np.uint32))
            np.testing.assert_array_equal(ex["vscale"][b, h].view(np.uint32), kv["sv"].view(np.uint32))
            if w.smooth_v:
                np.testing.assert_array_equal(ex["vmean"][b, h].view(np.uint32), kv["vbar"].view(np.uint32))
            np.testing.assert_array_equal(ex16["v16"][b, h].astype(np.float64), kv["v4"])


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_fp4_output_matches_online_form(w):
    g = _run(w)
    ref = sage_attention(g["qn"], g["kn"], g["vn"], pv="fp4", p_max="running", **oracle_kw(w))
    o = g["o"]
    assert np.isfinite(o).all()
    assert max_abs_excess(o, ref["o"], w.dtype) <= TOL4_ONLINE_MAX_ABS
    assert excess_fraction(o, ref["o"], w.dtype, TOL4_ONLINE_ELEM) <= TOL4_ONLINE_ELEM_FRAC
    assert cosine(o, ref["o"]) >= TOL4_ONLINE_COS
    if w.return_lse:
        assert np.abs(g["lse"] - ref["lse"]).max() <= TOL4_ONLINE_LSE


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_fp4_output_within_tolerance(w):
    g = _run(w)
    ref = sage_attention(g["qn"], g["kn"], g["vn"], pv="fp4", **oracle_kw(w))
    o = g["o"]
    assert max_abs_excess(o, ref["o"], w.dtype) <= TOL4_FINAL_MAX_ABS
    assert cosine(o, ref["o"]) >= TOL4_FINAL_COS
    grp = w.Hq // w.Hkv
    for b in range(w.B):
        for h in range(w.Hq):
            of, _ = attention_fp64(g["qn"][b, h], g["kn"][b, h // grp], g["vn"][b, h // grp],
                                   ref["sm_scale"], w.is_causal)
            assert cosine(o[b, h], of) >= TOL4_COS_FP64
    if w.return_lse:
        assert np.abs(g["lse"] - ref["lse"]).max() <= TOL4_LSE


def test_fp4_full_size_sampled_rows():
    # the DiT shape's head geometry (17776 keys, d = 64, the 112-row tail) on two heads;
    # sampled query rows across the tiles, including the tail tile
    import quantized_attention_mean_gb300 as qa
    w = Workload("dit_fp4_h2", 1, 2, 2, 17776, 17776, 64, dtype="bf16", gran="per_warp",
                 accum="fp16+fp32", smooth_v=True, k_offset_std=4.0, v_offset_std=2.0,
                 return_lse=True)
    q, k, v = dense_inputs(w, 3)
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    dev = torch.device("cuda:0")
    ws = qa.alloc_workspace(qa.workspace_bytes(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran), dev)
    out, lse = qa.sage_attn_fp4(q.to(dev), k.to(dev), v.to(dev), workspace=ws, **gpu_kw(w))
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    rows = np.array([0, 1, 127, 128, 4097, 9000, 17663, 17664, 17700, 17775])
    ref = sage_attention(qn, kn, vn, pv="fp4", p_max="running", rows=rows, **oracle_kw(w))
    o = out_to_hnd(out, w.layout)[:, :, rows]
    assert max_abs_excess(o, ref["o"], w.dtype) <= TOL4_ONLINE_MAX_ABS
    assert cosine(o, ref["o"]) >= TOL4_ONLINE_COS
    assert np.abs(lse.cpu().numpy()[:, :, rows] - ref["lse"]).max() <= TOL4_ONLINE_LSE
