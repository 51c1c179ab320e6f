"""GPU parity of the FP16 P·V variant (sage_attn_qk_int8_pv_fp16) against the oracle's
pv="fp16" emulation, on the shapes of the main parity suite."""

import numpy as np
import pytest
import torch

from helpers import (TOL_COS, TOL_COS_FP64, TOL_LSE, TOL_MAX_ABS, assert_online_parity, cosine, gpu_kw,
                     max_abs_excess, oracle_kw, out_to_hnd)
from oracle.attention import attention_fp64, sage_attention
from quantized_attention_mean_gb300.workloads import WORKLOADS, Workload, dense_inputs, to_hnd_f32

pytestmark = pytest.mark.gpu

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
    Workload("fp16acc_d128", 1, 2, 2, 512, 512, 128, gran="per_warp", accum="fp16+fp32"),
    Workload("pad_d72", 1, 2, 1, 140, 260, 72, dtype="bf16", gran="per_thread", accum="fp32+fp32"),
    Workload("tail_pair_long_keys", 1, 2, 2, 300, 1100, 64, dtype="bf16", gran="per_thread",
             smooth_v=True, v_offset_std=1.0),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_pv16_output_within_tolerance(w):
    import quantized_attention_mean_gb300 as qa
    q, k, v = dense_inputs(w, 0)
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    ref = sage_attention(qn, kn, vn, pv="fp16", **oracle_kw(w))
    dev = torch.device("cuda:0")
    ws = qa.alloc_workspace(qa.workspace_bytes(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran), dev)
    res = qa.sage_attn_qk_int8_pv_fp16(q.to(dev), k.to(dev), v.to(dev), workspace=ws, **gpu_kw(w))
    out, lse = res if w.return_lse else (res, None)
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    o = out_to_hnd(out, w.layout)
    assert np.isfinite(o).all()
    assert max_abs_excess(o, ref["o"], w.dtype) <= TOL_MAX_ABS
    assert cosine(o, ref["o"]) >= TOL_COS
    grp = w.Hq // w.Hkv
    for b in range(w.B):
        for h in range(w.Hq):
            of, _ = attention_fp64(qn[b, h], kn[b, h // grp], vn[b, h // grp], ref["sm_scale"], w.is_causal)
            assert cosine(o[b, h], of) >= TOL_COS_FP64
    if w.return_lse:
        assert np.max(np.abs(lse.cpu().numpy() - ref["lse"])) <= TOL_LSE


def test_pv16_more_accurate_than_fp8_on_the_gpu():
    # the fallback's purpose: closer to exact attention than the FP8 P·V path
    import quantized_attention_mean_gb300 as qa
    w = Workload("acc_cmp", 1, 4, 4, 512, 512, 128, gran="per_thread", accum="fp32")
    q, k, v = dense_inputs(w, 1)
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    dev = torch.device("cuda:0")
    o16 = out_to_hnd(qa.sage_attn_qk_int8_pv_fp16(q.to(dev), k.to(dev), v.to(dev), **gpu_kw(w)), w.layout)
    o8 = out_to_hnd(qa.sage_attn(q.to(dev), k.to(dev), v.to(dev), **gpu_kw(w)), w.layout)
    sm = 1.0 / np.sqrt(128.0)
    exact = np.stack([attention_fp64(qn[0, h], kn[0, h], vn[0, h], sm, False)[0] for h in range(4)])
    assert np.abs(o16[0] - exact).max() < np.abs(o8[0] - exact).max()


def test_pv16_full_size_sampled_rows():
    # the DiT shape's head geometry (17776 keys, d = 64, 139 key tiles with the 112-row tail) on
    # two heads; sampled query rows across the tiles, against the oracle's online form
    import quantized_attention_mean_gb300 as qa
    w = Workload("dit_pv16_h2", 1, 2, 2, 17776, 17776, 64, dtype="bf16", gran="per_warp",
                 accum="fp16+fp32", smooth_v=True, k_offset_std=4.0, v_offset_std=2.0,
                 return_lse=True)
    q, k, v = dense_inputs(w, 4)
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    dev = torch.device("cuda:0")
    ws = qa.alloc_workspace(qa.workspace_bytes(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran), dev)
    out, lse = qa.sage_attn_qk_int8_pv_fp16(q.to(dev), k.to(dev), v.to(dev), workspace=ws, **gpu_kw(w))
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    rows = np.array([0, 1, 127, 128, 4097, 9000, 17663, 17664, 17700, 17775])
    ref = sage_attention(qn, kn, vn, pv="fp16", p_max="running", rows=rows, **oracle_kw(w))
    o = out_to_hnd(out, w.layout)[:, :, rows]
    assert_online_parity(o, ref["o"], w.dtype, lse.cpu().numpy()[:, :, rows], ref["lse"])
