"""Bounded device waits: with the producer told to issue no K/V loads (a flag nothing
else sets), every consumer wait in the attention kernel runs into its ~2 s bound; the kernel
exits cleanly, the workspace status reads SAGE_ERR_TIMEOUT, and the CUDA context stays usable.
No GPU fault, trap or unbounded wait is involved. Covered for both head dims (rotating S
buffers with two issuers at 64, one S buffer per tile with the s_free trigger at 128), each
P·V format, and CTAs with one query tile as well as two."""

import pytest
import torch

pytestmark = pytest.mark.gpu

CASES = [(64, "fp8", 200), (64, "fp16", 200), (64, "fp4", 200), (64, "fp8", 100),
         (128, "fp8", 200), (128, "fp16", 200), (128, "fp4", 100)]


@pytest.mark.parametrize("d,pv,n", CASES, ids=[f"d{d}-{pv}-n{n}" for d, pv, n in CASES])
def test_stalled_producer_times_out_cleanly(d, pv, n):
    import quantized_attention_mean_gb300 as qa
    from quantized_attention_mean_gb300 import _lib
    lib = _lib.load()
    dev = torch.device("cuda:0")
    fn = {"fp8": qa.sage_attn, "fp16": qa.sage_attn_qk_int8_pv_fp16, "fp4": qa.sage_attn_fp4}[pv]
    q = torch.randn(1, 2, n, d, device=dev, dtype=torch.float16)
    ws = qa.alloc_workspace(qa.workspace_bytes(1, 2, 2, n, n, d), dev)
    try:
        assert lib.sage_debug_stall_attention(1) == 0
        fn(q, q, q, workspace=ws)
        assert qa.read_device_status(ws) == 9          # SAGE_ERR_TIMEOUT
    finally:
        lib.sage_debug_stall_attention(0)
    out = fn(q, q, q, workspace=ws)
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    assert torch.isfinite(out.float()).all()
