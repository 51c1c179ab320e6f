"""Full-size workloads, in the launch configuration bench.py times: every head's quantised
tensors (INT8 Q / K codes and scales, E4M3 V codes and scales, the smoothing means) bit for
bit, and sampled query rows of three heads against the oracle's attention (which computes
those rows one by one).

Workloads: 4K self-attention (2x8x4096^2, d=128, fp16+fp32), causal GQA decoder (1x32/8x8192^2,
bf16 NHD, per_thread, LSE), video-DiT long sequence (2x48x17776^2, d=64, biased K/V,
smooth_v, fp16+fp32: 138 full tiles + a 112-row tail), ragged varlen batch (16 sequences,
lengths uniform in [128, 8192])."""

import numpy as np
import pytest
import torch

from oracle.attention import attend_head, quantize_kv_head, quantize_q_head, sage_attention_varlen, default_sm_scale
from quantized_attention_mean_gb300.workloads import (ACC, GRAN, WORKLOADS, dense_inputs, to_hnd_f32,
                                                      varlen_inputs)

from helpers import (TOL_COS, TOL_LSE, TOL_MAX_ABS, assert_online_parity, cosine, max_abs_excess,
                     out_to_hnd, run_gpu_dense)

pytestmark = pytest.mark.gpu


def _rows(n):
    rng = np.random.default_rng(n)
    r = set([0, 1, 127, 128, n // 2, n - 1, n - 2]) | set(rng.integers(0, n, 25).tolist())
    return np.array(sorted(x for x in r if 0 <= x < n))


@pytest.mark.parametrize("name", ["sdpa4k", "gqa_causal8k", "dit17776"])
def test_full_size_dense_sampled(name):
    import quantized_attention_mean_gb300 as qa
    w = WORKLOADS[name]
    q, k, v = dense_inputs(w, 0)
    g = run_gpu_dense(w, q, k, v)
    assert g["status"] == 0
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    del q, k, v
    o = out_to_hnd(g["out"], w.layout)
    assert np.isfinite(o).all()
    lse = g["lse"].cpu().numpy() if w.return_lse else None
    ex = {n: t.cpu().numpy() for n, t in
          qa.export_quant(g["ws"], w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran).items()}
    grp = w.Hq // w.Hkv
    gran = GRAN[w.gran]
    # every head's quantised tensors, bit for bit: K / V codes, scales and means per KV head,
    # Q codes and scales per query head
    rows = _rows(w.Nq)
    heads = [(0, 0), (w.B - 1, w.Hq - 1), (0, w.Hq // 2 + 1)]
    kvq_keep = {}
    for b in range(w.B):
        for hk in range(w.Hkv):
            kvq = quantize_kv_head(kn[b, hk], vn[b, hk], gran, w.smooth_k, w.smooth_v)
            np.testing.assert_array_equal(ex["k8"][b, hk], kvq["k8"])
            np.testing.assert_array_equal(ex["v8"][b, hk], kvq["v8"])
            np.testing.assert_array_equal(ex["sk"][b, hk].view(np.uint32), kvq["sk"].view(np.uint32))
            np.testing.assert_array_equal(ex["vscale"][b, hk].view(np.uint32), kvq["sv"].view(np.uint32))
            np.testing.assert_array_equal(ex["kmean"][b, hk].view(np.uint32), kvq["kbar"].view(np.uint32))
            np.testing.assert_array_equal(ex["vmean"][b, hk].view(np.uint32), kvq["vbar"].view(np.uint32))
            if any((b, hk) == (hb, hh // grp) for hb, hh in heads):
                kvq_keep[(b, hk)] = kvq
        for h in range(w.Hq):
            qq = quantize_q_head(qn[b, h], gran)
            np.testing.assert_array_equal(ex["q8"][b, h], qq["q8"])
            np.testing.assert_array_equal(ex["sq"][b, h].view(np.uint32), qq["sq"].view(np.uint32))
    del ex
    # sampled rows of three heads against the oracle's attention
    sm = default_sm_scale(w.d)
    for (b, h) in heads:
        kvq = kvq_keep[(b, h // grp)]
        qq = quantize_q_head(qn[b, h], gran)
        ref = attend_head(qn[b, h], kvq, gran=gran, sm_scale=sm, is_causal=w.is_causal,
                          accum=ACC[w.accum], rows=rows, qq=qq)
        got = o[b, h, rows]
        assert max_abs_excess(got, ref["o"], w.dtype) <= TOL_MAX_ABS
        assert cosine(got, ref["o"]) >= TOL_COS
        if lse is not None:
            assert np.abs(lse[b, h, rows] - ref["lse"]).max() <= TOL_LSE
        # the online form over every key tile of the full sequence
        onl = attend_head(qn[b, h], kvq, gran=gran, sm_scale=sm, is_causal=w.is_causal,
                          accum=ACC[w.accum], rows=rows, qq=qq, p_max="running")
        assert_online_parity(got, onl["o"], w.dtype, lse[b, h, rows] if lse is not None else None,
                             onl["lse"])


def test_full_size_varlen_sampled():
    import quantized_attention_mean_gb300 as qa
    w = WORKLOADS["varlen16"]
    q, k, v, cu_q, cu_k, lens = varlen_inputs(w, 0)
    dev = torch.device("cuda:0")
    ws = qa.alloc_workspace(qa.varlen_workspace_bytes(len(lens), w.Hq, w.Hkv, q.shape[0], k.shape[0],
                                                      w.d, w.gran), dev)
    out = qa.sage_attn_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev), max(lens),
                              max(lens), qk_quant_gran=w.gran, pv_accum_dtype=w.accum,
                              smooth_k=w.smooth_k, smooth_v=w.smooth_v, workspace=ws)
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    qn, kn, vn = (t.float().numpy() for t in (q, k, v))
    cu = cu_q.numpy()
    sm = default_sm_scale(w.d)
    for b in (0, int(np.argmax(lens)), len(lens) - 1):
        sl = slice(cu[b], cu[b + 1])
        for h in (0, w.Hq - 1):
            kvq = quantize_kv_head(kn[sl, h], vn[sl, h], GRAN[w.gran], w.smooth_k, w.smooth_v)
            rows = _rows(lens[b])
            ref = attend_head(qn[sl, h], kvq, gran=GRAN[w.gran], sm_scale=sm, is_causal=False,
                              accum=ACC[w.accum], rows=rows)
            got = o[sl, h][rows]
            assert max_abs_excess(got, ref["o"], w.dtype) <= TOL_MAX_ABS
            assert cosine(got, ref["o"]) >= TOL_COS
            onl = attend_head(qn[sl, h], kvq, gran=GRAN[w.gran], sm_scale=sm, is_causal=False,
                              accum=ACC[w.accum], rows=rows, p_max="running")
            assert_online_parity(got, onl["o"], w.dtype)
