"""The Python binding's argument checks, on the CPU (they run before any device work). The C
ABI sees only pointers and strides, so tensors whose shapes disagree (a v smaller than k, an
out or lse smaller than q's) must be rejected here; so must tensors that are not on a CUDA
device."""

import pytest
import torch

import quantized_attention_mean_gb300 as qa


def _t(*shape, dtype=torch.float16):
    return torch.zeros(shape, dtype=dtype)


def test_dense_argument_checks():
    q, k = _t(1, 2, 64, 64), _t(1, 2, 80, 64)
    with pytest.raises(ValueError, match="v must have k's shape"):
        qa.sage_attn(q, k, _t(1, 2, 79, 64))
    with pytest.raises(ValueError, match="batch size and head_dim"):
        qa.sage_attn(q, _t(2, 2, 80, 64), _t(2, 2, 80, 64))
    with pytest.raises(ValueError, match="batch size and head_dim"):
        qa.sage_attn(q, _t(1, 2, 80, 32), _t(1, 2, 80, 32))
    with pytest.raises(ValueError, match="4-D"):
        qa.sage_attn(_t(2, 64, 64), k, k)
    with pytest.raises(TypeError):
        qa.sage_attn(q, k, _t(1, 2, 80, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="tensor_layout"):
        qa.sage_attn(q, k, k, tensor_layout="BHSD")
    with pytest.raises(ValueError, match="out must"):
        qa.sage_attn(q, k, k, out=_t(1, 2, 63, 64))
    with pytest.raises(ValueError, match="lse must"):
        qa.sage_attn(q, k, k, return_lse=True, lse=torch.zeros(1, 2, 63))
    with pytest.raises(ValueError, match="lse must"):
        qa.sage_attn(q, k, k, return_lse=True, lse=torch.zeros(1, 2, 64, dtype=torch.float16))
    with pytest.raises(ValueError, match="CUDA device"):
        qa.sage_attn(q, k, k)                       # consistent, but on the CPU
    with pytest.raises(ValueError, match="v must have k's shape"):
        qa.sage_attn_qk_int8_pv_fp16(q, k, _t(1, 1, 80, 64))


def test_varlen_argument_checks():
    q, k = _t(100, 2, 64), _t(120, 2, 64)
    cu = torch.tensor([0, 40, 100], dtype=torch.int32)
    cu_k = torch.tensor([0, 60, 120], dtype=torch.int32)
    with pytest.raises(ValueError, match="v must have k's shape"):
        qa.sage_attn_varlen(q, k, _t(119, 2, 64), cu, cu_k, 60, 60)
    with pytest.raises(ValueError, match="3-D"):
        qa.sage_attn_varlen(_t(1, 100, 2, 64), k, k, cu, cu_k, 60, 60)
    with pytest.raises(ValueError, match="cu_seqlens_q and cu_seqlens_k"):
        qa.sage_attn_varlen(q, k, k, cu, cu_k[:2], 60, 60)
    with pytest.raises(ValueError, match="cu_seqlens_q and cu_seqlens_k"):
        qa.sage_attn_varlen(q, k, k, cu.view(1, 3), cu_k.view(1, 3), 60, 60)
    with pytest.raises(TypeError):
        qa.sage_attn_varlen(q, k, k, cu.long(), cu_k, 60, 60)
    with pytest.raises(ValueError, match="out must"):
        qa.sage_attn_varlen(q, k, k, cu, cu_k, 60, 60, out=_t(99, 2, 64))
    with pytest.raises(ValueError, match="lse must"):
        qa.sage_attn_varlen(q, k, k, cu, cu_k, 60, 60, return_lse=True, lse=torch.zeros(100, 2))
    with pytest.raises(ValueError, match="CUDA device"):
        qa.sage_attn_varlen(q, k, k, cu, cu_k, 60, 60)


def test_merge_argument_checks():
    o = [_t(1, 2, 8, 64), _t(1, 2, 8, 64)]
    l = [torch.zeros(1, 2, 8), torch.zeros(1, 2, 8)]
    with pytest.raises(ValueError, match="out must"):
        qa.merge_partials(o, l, out=_t(1, 2, 7, 64))
    with pytest.raises(ValueError, match="lse must"):
        qa.merge_partials(o, l, lse=torch.zeros(1, 2, 7))
    with pytest.raises(ValueError, match="CUDA device"):
        qa.merge_partials(o, l)
