"""sage_attn_no_alloc: the dense forward for callers that cannot allocate device memory
(for example a plugin that runs inside a host engine which owns all device memory and
forbids allocation while it executes). It takes its scratch from an array built into the
library instead of a caller workspace. This file is collected last, so a run that stops at
its first failure has already run every other test.

Checked through the C ABI against sage_attn on two calls in a row (different sizes and
options, so a stale scratch from the first call would show). Both run the same kernels on the
same inputs and the pipeline is deterministic (integer statistics sums, fixed launch order), so
the outputs and LSE must agree bit for bit; and the size limit's error."""

import ctypes

import pytest
import torch

from quantized_attention_mean_gb300.workloads import Workload, dense_inputs


pytestmark = pytest.mark.gpu

CALLS = [
    Workload("first", 2, 4, 2, 300, 300, 128, gran="per_warp", accum="fp32", return_lse=True),
    Workload("second", 1, 2, 2, 500, 260, 64, dtype="bf16", layout="NHD", is_causal=True,
             gran="per_thread", accum="fp16+fp32", smooth_v=True, v_offset_std=2.0),
]


def _no_alloc(lib, q, k, v, out, lse, w):
    import quantized_attention_mean_gb300 as qa
    from quantized_attention_mean_gb300 import _tensor, DTYPE, GRAN, ACC, LAYOUT
    st = lib.sage_attn_no_alloc(
        ctypes.byref(_tensor(q)), ctypes.byref(_tensor(k)), ctypes.byref(_tensor(v)),
        ctypes.byref(_tensor(out)), ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
        w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, DTYPE[q.dtype], LAYOUT[w.layout], int(w.is_causal),
        float("nan"), int(w.return_lse), GRAN[w.gran], ACC[w.accum], int(w.smooth_k),
        int(w.smooth_v), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_no_alloc_matches_sage_attn_on_consecutive_calls():
    import quantized_attention_mean_gb300 as qa
    from quantized_attention_mean_gb300 import _lib
    lib = _lib.load()
    dev = torch.device("cuda:0")
    for w in CALLS:
        q, k, v = (t.to(dev) for t in dense_inputs(w, seed=3))
        ref = qa.sage_attn(q, k, v, tensor_layout=w.layout, is_causal=w.is_causal,
                           return_lse=w.return_lse, qk_quant_gran=w.gran, pv_accum_dtype=w.accum,
                           smooth_k=w.smooth_k, smooth_v=w.smooth_v)
        ref_o, ref_l = ref if w.return_lse else (ref, None)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq, w.Nq), float("nan"), device=dev) if w.return_lse else None
        assert _no_alloc(lib, q, k, v, out, lse, w) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref_o)
        if lse is not None:
            assert torch.equal(lse, ref_l)


def test_no_alloc_rejects_problems_beyond_its_scratch():
    from quantized_attention_mean_gb300 import _lib
    lib = _lib.load()
    dev = torch.device("cuda:0")
    w = Workload("big", 4, 32, 32, 4096, 4096, 128)  # needs far more than 32 MiB of scratch
    assert lib.sage_attn_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, 1) > (32 << 20)
    q = torch.zeros((1, 1, 1, 128), dtype=torch.float16, device=dev)  # never read
    out = torch.empty_like(q)
    assert _no_alloc(lib, q, q, q, out, None, w) == 6  # SAGE_ERR_WORKSPACE
