"""The scaled_dot_product_attention stand-in: argument handling on the host, and on the GPU
the same result as sage_attn plus closeness to torch's own attention."""

import pytest
import torch

import quantized_attention_mean_gb300 as qa
from helpers import TOL_COS_FP64, cosine


def test_rejects_what_the_method_does_not_support():
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(NotImplementedError):
        qa.scaled_dot_product_attention(q, q, q, attn_mask=torch.ones(8, 8, dtype=torch.bool))
    with pytest.raises(NotImplementedError):
        qa.scaled_dot_product_attention(q, q, q, dropout_p=0.1)
    with pytest.raises(ValueError):
        qa.scaled_dot_product_attention(q, q[:, :, :, :, None], q)
    with pytest.raises(ValueError):
        qa.scaled_dot_product_attention(q, torch.zeros(1, 3, 8, 64, dtype=torch.float16), q)


@pytest.mark.gpu
@pytest.mark.parametrize("shape_q,shape_kv,causal,dtype", [
    ((2, 8, 300, 128), (2, 2, 300, 128), True, torch.bfloat16),
    ((4, 200, 64), (4, 333, 64), False, torch.float16),
])
def test_matches_sage_attn_and_torch(shape_q, shape_kv, causal, dtype):
    g = torch.Generator().manual_seed(3)
    dev = torch.device("cuda:0")
    q = torch.randn(shape_q, generator=g).to(dtype).to(dev)
    k = torch.randn(shape_kv, generator=g).to(dtype).to(dev)
    v = torch.randn(shape_kv, generator=g).to(dtype).to(dev)
    o = qa.scaled_dot_product_attention(q, k, v, is_causal=causal)
    batched = q.dim() == 4
    q4, k4, v4 = (t if batched else t.unsqueeze(0) for t in (q, k, v))
    o_direct = qa.sage_attn(q4, k4, v4, is_causal=causal)
    assert torch.equal(o if batched else o.unsqueeze(0), o_direct)
    rep = q4.shape[1] // k4.shape[1]
    ref = torch.nn.functional.scaled_dot_product_attention(
        q4.double(), k4.double().repeat_interleave(rep, 1), v4.double().repeat_interleave(rep, 1),
        is_causal=causal)
    assert cosine(o_direct.double().cpu().numpy(), ref.cpu().numpy()) >= TOL_COS_FP64
