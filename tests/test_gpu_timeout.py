"""Bounded device waits: with the producer told to issue no K/V loads (a flag nothing
else sets), every consumer wait in the attention kernel runs into its ~2 s bound; the kernel
exits cleanly, the workspace status reads SAGE_ERR_TIMEOUT, and the CUDA context stays usable.
No GPU fault, trap or unbounded wait is involved."""

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_stalled_producer_times_out_cleanly():
    import quantized_attention_mean_gb300 as qa
    from quantized_attention_mean_gb300 import _lib
    lib = _lib.load()
    dev = torch.device("cuda:0")
    q = torch.randn(1, 2, 200, 64, device=dev, dtype=torch.float16)
    ws = qa.alloc_workspace(qa.workspace_bytes(1, 2, 2, 200, 200, 64), dev)
    try:
        assert lib.sage_debug_stall_attention(1) == 0
        qa.sage_attn(q, q, q, workspace=ws)
        assert qa.read_device_status(ws) == 9          # SAGE_ERR_TIMEOUT
    finally:
        lib.sage_debug_stall_attention(0)
    out = qa.sage_attn(q, q, q, workspace=ws)
    torch.cuda.synchronize()
    assert qa.read_device_status(ws) == 0
    assert torch.isfinite(out.float()).all()
