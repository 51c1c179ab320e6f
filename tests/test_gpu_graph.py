"""The entry points are capturable into a CUDA graph: no host synchronisation, allocation or
host-side read of device data inside a call. A graph of several calls (dense, FP16 P·V and
varlen), replayed, gives the same bytes as the direct calls and leaves the status clear; the
default path choice for short problems (short-sequence kernel when called directly, the main
pipeline when captured) is checked against each implementation selected explicitly."""

import pytest
import torch

from quantized_attention_mean_gb300.workloads import Workload, dense_inputs, varlen_inputs

from helpers import gpu_kw

pytestmark = pytest.mark.gpu


def _dense_call(qa, w, q, k, v, out, lse, ws, pv16):
    fn = qa.sage_attn_qk_int8_pv_fp16 if pv16 else qa.sage_attn
    fn(q, k, v, out=out, lse=lse, workspace=ws, **gpu_kw(w))


@pytest.mark.parametrize("pv16", [False, True])
def test_dense_graph_replay_matches_direct_calls(pv16):
    import quantized_attention_mean_gb300 as qa
    dev = torch.device("cuda:0")
    w = Workload("graph_dense", 2, 4, 2, 300, 333, 128, dtype="bf16", layout="NHD", is_causal=True,
                 gran="per_thread", accum="fp32", return_lse=True, k_offset_std=3.0)
    q, k, v = (t.to(dev) for t in dense_inputs(w, 3))
    ws = qa.alloc_workspace(qa.workspace_bytes(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran), dev)
    out, lse = torch.empty_like(q), torch.empty(w.B, w.Hq, w.Nq, device=dev)
    _dense_call(qa, w, q, k, v, out, lse, ws, pv16)
    torch.cuda.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _dense_call(qa, w, q, k, v, out, lse, ws, pv16)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            _dense_call(qa, w, q, k, v, out, lse, ws, pv16)
    out.zero_()
    lse.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_l.view(torch.int32))


def test_varlen_graph_replay_matches_direct_call():
    import quantized_attention_mean_gb300 as qa
    dev = torch.device("cuda:0")
    w = Workload("graph_varlen", 3, 4, 4, 0, 0, 64, gran="per_warp", accum="fp16+fp32", varlen=True,
                 n_seqs=3, return_lse=True)
    q, k, v, cu, _, lens = varlen_inputs(w, 0, [200, 7, 390])
    q, k, v, cu = (t.to(dev) for t in (q, k, v, cu))
    ws = qa.alloc_workspace(qa.varlen_workspace_bytes(len(lens), w.Hq, w.Hkv, q.shape[0], k.shape[0],
                                                      w.d, w.gran), dev)
    out = torch.empty_like(q)
    lse = torch.empty(w.Hq, q.shape[0], device=dev)

    def call():
        qa.sage_attn_varlen(q, k, v, cu, cu, max(lens), max(lens), return_lse=True, qk_quant_gran=w.gran,
                            pv_accum_dtype=w.accum, out=out, lse=lse, workspace=ws)

    call()
    torch.cuda.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_l.view(torch.int32))


def test_auto_path_direct_short_captured_main():
    # a short head_dim-64 problem: called directly the default path runs the short-sequence
    # kernel (same bytes as selecting it), captured into a graph it runs the main pipeline
    # (same bytes as selecting that)
    import quantized_attention_mean_gb300 as qa
    dev = torch.device("cuda:0")
    w = Workload("auto_path", 1, 4, 2, 300, 200, 64, dtype="bf16", gran="per_warp", accum="fp32",
                 return_lse=True, smooth_v=True)
    q, k, v = (t.to(dev) for t in dense_inputs(w, 4))
    ws = qa.alloc_workspace(qa.workspace_bytes(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.gran), dev)
    out, lse = torch.empty_like(q), torch.empty(w.B, w.Hq, w.Nq, device=dev)
    res = {}
    try:
        for path in ("main", "short", "auto"):
            qa.select_path(path)
            _dense_call(qa, w, q, k, v, out, lse, ws, False)
            torch.cuda.synchronize()
            res[path] = (out.clone(), lse.clone())
        qa.select_path("auto")
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            _dense_call(qa, w, q, k, v, out, lse, ws, False)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            _dense_call(qa, w, q, k, v, out, lse, ws, False)
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
    finally:
        qa.select_path("auto")
    assert qa.read_device_status(ws) == 0
    same = lambda a, b: (torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
                         and torch.equal(a[1].view(torch.int32), b[1].view(torch.int32)))
    assert same(res["auto"], res["short"])
    assert same((out, lse), res["main"])
    assert not same(res["main"], res["short"])  # the two implementations round differently
