"""GPU parity of sage_merge_partials (composition of partial results over disjoint key sets,
the log-sum-exp use the method names for ring-style attention) against oracle.merge."""

import numpy as np
import pytest
import torch

from helpers import TOL_COS, TOL_MAX_ABS, cosine, max_abs_excess, oracle_kw, out_to_hnd
from oracle.attention import sage_attention
from oracle.merge import merge_partials as oracle_merge
from quantized_attention_mean_gb300.workloads import Workload, dense_inputs, to_hnd_f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,layout,n,d", [("fp16", "HND", 1, 64), ("fp16", "HND", 3, 128),
                                              ("bf16", "NHD", 5, 128), ("bf16", "HND", 2, 72),
                                              ("fp16", "NHD", 16, 32)])
def test_merge_kernel_matches_oracle(dtype, layout, n, d):
    import quantized_attention_mean_gb300 as qa
    g = torch.Generator().manual_seed(n * 1000 + d)
    B, H, N = 2, 3, 77
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    shape = (B, H, N, d) if layout == "HND" else (B, N, H, d)
    outs = [(torch.randn(shape, generator=g) * 2).to(tdt) for _ in range(n)]
    lses = [torch.randn((B, H, N), generator=g) * 3 + 5 for _ in range(n)]
    if n > 1:
        lses[1][0, 1, :10] = -float("inf")           # a part that saw no key for some rows
    lses[0][1, 2, 5] = -float("inf")
    if n == 1:
        pass
    else:
        for l in lses:
            l[1, 0, 3] = -float("inf")               # a row no part sees
    dev = torch.device("cuda:0")
    o, lse = qa.merge_partials([x.to(dev) for x in outs], [l.to(dev) for l in lses], tensor_layout=layout)
    torch.cuda.synchronize()
    hnd = lambda t: (t.float().numpy() if layout == "HND" else t.float().transpose(1, 2).numpy())
    o_ref, lse_ref = oracle_merge([hnd(x) for x in outs], [l.numpy() for l in lses])
    o_gpu = hnd(o.cpu())
    assert max_abs_excess(o_gpu, o_ref, dtype) <= 1e-4
    lg = lse.cpu().numpy()
    fin = np.isfinite(lse_ref)
    np.testing.assert_array_equal(np.isfinite(lg), fin)
    np.testing.assert_allclose(lg[fin], lse_ref[fin], atol=2e-5, rtol=0)
    if n > 1:
        assert (o_gpu[1, 0, 3] == 0).all()


def test_merge_in_place_into_first_part():
    import quantized_attention_mean_gb300 as qa
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(7)
    outs = [torch.randn((1, 2, 40, 64), generator=g).half().to(dev) for _ in range(3)]
    lses = [torch.randn((1, 2, 40), generator=g).to(dev) for _ in range(3)]
    ref, ref_lse = qa.merge_partials(outs, lses)
    first = outs[0].clone()
    qa.merge_partials([first] + outs[1:], lses, out=first)
    torch.cuda.synchronize()
    assert torch.equal(first, ref)


@pytest.mark.parametrize("w,cuts", [
    (Workload("ring_hnd", 1, 4, 2, 300, 520, 128, gran="per_warp", accum="fp32", return_lse=True,
              k_offset_std=3.0), [128, 384]),
    (Workload("ring_nhd_bf16", 2, 2, 2, 200, 333, 64, dtype="bf16", layout="NHD", gran="per_thread",
              accum="fp16+fp32", smooth_v=True, return_lse=True, v_offset_std=2.0), [100]),
])
def test_ring_composition_matches_oracle(w, cuts):
    # attention over K/V chunks (each a full sage_attn call with return_lse), merged on the
    # GPU, against the oracle's per-chunk results merged in float64
    import quantized_attention_mean_gb300 as qa
    q, k, v = dense_inputs(w, 0)
    qn, kn, vn = (to_hnd_f32(t, w.layout) for t in (q, k, v))
    dev = torch.device("cuda:0")
    tok = 2 if w.layout == "HND" else 1
    bounds = [0] + cuts + [w.Nk]
    outs, lses, o_parts, l_parts = [], [], [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        kc, vc = k.narrow(tok, a, b - a).contiguous(), v.narrow(tok, a, b - a).contiguous()
        o, l = qa.sage_attn(q.to(dev), kc.to(dev), vc.to(dev), tensor_layout=w.layout,
                            return_lse=True, qk_quant_gran=w.gran, pv_accum_dtype=w.accum,
                            smooth_k=w.smooth_k, smooth_v=w.smooth_v)
        outs.append(o)
        lses.append(l)
        ref = sage_attention(qn, kn[:, :, a:b], vn[:, :, a:b], **oracle_kw(w))
        o_parts.append(ref["o"])
        l_parts.append(ref["lse"])
    o, lse = qa.merge_partials(outs, lses, tensor_layout=w.layout)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_merge(o_parts, l_parts)
    o_gpu = out_to_hnd(o, w.layout)
    assert max_abs_excess(o_gpu, o_ref, w.dtype) <= TOL_MAX_ABS
    assert cosine(o_gpu, o_ref) >= TOL_COS
    assert np.max(np.abs(lse.cpu().numpy() - lse_ref)) <= 2e-2
