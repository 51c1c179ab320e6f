"""GPU parity of the variable-length path (sageattn_varlen: cu_seqlens_q / cu_seqlens_k)
against the oracle run per sequence, plus device-side cu_seqlens validation."""

import numpy as np
import pytest
import torch

from oracle.attention import attention_fp64, sage_attention_varlen
from quantized_attention_mean_gb300.workloads import ACC, GRAN, Workload, varlen_inputs

from helpers import (TOL_COS, TOL_COS_FP64, TOL_LSE, TOL_MAX_ABS, assert_online_parity, cosine,
                     max_abs_excess)

pytestmark = pytest.mark.gpu

CASES = [
    (Workload("vl_basic", 5, 4, 4, 0, 0, 128, gran="per_warp", accum="fp32", varlen=True, n_seqs=5,
              return_lse=True), [5, 130, 1, 64, 300]),
    (Workload("vl_causal_gqa", 4, 8, 2, 0, 0, 64, dtype="bf16", is_causal=True, gran="per_thread",
              accum="fp32", varlen=True, n_seqs=4, return_lse=True, k_offset_std=3.0), [256, 17, 129, 200]),
    (Workload("vl_empty_seq", 3, 2, 2, 0, 0, 72, gran="per_block", accum="fp16+fp32", smooth_v=True,
              varlen=True, n_seqs=3, v_offset_std=2.0), [40, 0, 90]),
]


def _run(w, lens, pv="fp8"):
    import quantized_attention_mean_gb300 as qa
    q, k, v, cu_q, cu_k, lens = varlen_inputs(w, 0, lens)
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    cqd, ckd = cu_q.to(dev), cu_k.to(dev)
    ws = qa.alloc_workspace(qa.varlen_workspace_bytes(len(lens), w.Hq, w.Hkv, q.shape[0], k.shape[0],
                                                      w.d, w.gran), dev)
    res = qa.sage_attn_varlen(qd, kd, vd, cqd, ckd, max(lens), max(lens), is_causal=w.is_causal,
                              return_lse=w.return_lse, qk_quant_gran=w.gran, pv_accum_dtype=w.accum,
                              smooth_k=w.smooth_k, smooth_v=w.smooth_v, workspace=ws, pv=pv)
    out, lse = res if w.return_lse else (res, None)
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    qn, kn, vn = (t.float().numpy() for t in (q, k, v))
    ref = sage_attention_varlen(qn, kn, vn, cu_q.numpy(), cu_k.numpy(), is_causal=w.is_causal,
                                gran=GRAN[w.gran], accum=ACC[w.accum], smooth_k=w.smooth_k,
                                smooth_v=w.smooth_v, pv=pv)
    return qn, kn, vn, cu_q.numpy(), out.float().cpu().numpy(), (lse.cpu().numpy() if lse is not None else None), ref


@pytest.mark.parametrize("pv", ["fp8", "fp16"])
@pytest.mark.parametrize("w,lens", CASES, ids=[c[0].name for c in CASES])
def test_varlen_parity(w, lens, pv):
    # pv="fp16": the FP16 P·V variant against the oracle's pv="fp16" emulation
    qn, kn, vn, cu, o, lse, ref = _run(w, lens, pv)
    assert np.isfinite(o).all()
    assert max_abs_excess(o, ref["o"], w.dtype) <= TOL_MAX_ABS
    assert cosine(o, ref["o"]) >= TOL_COS
    grp = w.Hq // w.Hkv
    sm = 1.0 / np.sqrt(w.d)
    for b in range(len(lens)):
        sl = slice(cu[b], cu[b + 1])
        if cu[b + 1] == cu[b]:
            continue
        for h in range(w.Hq):
            of, _ = attention_fp64(qn[sl, h], kn[sl, h // grp], vn[sl, h // grp], np.float32(sm), w.is_causal)
            assert cosine(o[sl, h], of) >= TOL_COS_FP64
    if lse is not None:
        assert np.abs(lse - ref["lse"]).max() <= TOL_LSE


@pytest.mark.parametrize("pv", ["fp8", "fp16"])
@pytest.mark.parametrize("w,lens", CASES, ids=[c[0].name for c in CASES])
def test_varlen_matches_online_form(w, lens, pv):
    # per sequence against the oracle's online form (P~ with the running maximum)
    qn, kn, vn, cu, o, lse, _ = _run(w, lens, pv)
    ref = sage_attention_varlen(qn, kn, vn, cu, cu, is_causal=w.is_causal, gran=GRAN[w.gran],
                                accum=ACC[w.accum], smooth_k=w.smooth_k, smooth_v=w.smooth_v,
                                pv=pv, p_max="running")
    assert_online_parity(o, ref["o"], w.dtype, lse, ref["lse"])


def test_varlen_bad_cu_seqlens_reports_status():
    import quantized_attention_mean_gb300 as qa
    dev = torch.device("cuda:0")
    q = torch.randn(100, 2, 64, device=dev, dtype=torch.float16)
    cu = torch.tensor([0, 60, 40, 100], dtype=torch.int32, device=dev)  # decreasing: invalid
    ws = qa.alloc_workspace(qa.varlen_workspace_bytes(3, 2, 2, 100, 100, 64), dev)
    qa.sage_attn_varlen(q, q, q, cu, cu, 100, 100, workspace=ws)
    assert qa.read_device_status(ws) == 12  # SAGE_ERR_SEQLENS
    # the context stays usable: a valid call afterwards succeeds
    cu2 = torch.tensor([0, 40, 60, 100], dtype=torch.int32, device=dev)
    qa.sage_attn_varlen(q, q, q, cu2, cu2, 40, 40, workspace=ws)
    assert qa.read_device_status(ws) == 0
