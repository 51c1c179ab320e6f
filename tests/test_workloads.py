"""The seeded input recipe both sides draw from (workloads.py): deterministic per seed; N(0, s)
with s the standard deviation; per-channel offsets of shape [Hkv, d] shared by every batch
entry and token; values rounded to the workload's dtype; HND / NHD as pure layouts; varlen
lengths uniform in the workload's range and packed with matching cu_seqlens. The metric's
operation count: 4·B·H·Nq·Nk·d, halved when causal, summed per sequence for varlen."""

import torch

from quantized_attention_mean_gb300.workloads import (WORKLOADS, Workload, dense_inputs,
                                                      to_hnd_f32, varlen_inputs, varlen_lengths)


def test_dense_inputs_are_deterministic_and_seeded():
    w = Workload("t", 2, 4, 2, 64, 96, 32, k_offset_std=3.0)
    a, b, c = dense_inputs(w, 0), dense_inputs(w, 0), dense_inputs(w, 1)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[0], c[0])
    q, k, v = a
    assert q.shape == (2, 4, 64, 32) and k.shape == (2, 2, 96, 32) and v.shape == (2, 2, 96, 32)
    assert q.dtype == torch.float16


def test_offsets_are_per_channel_and_shared():
    w = Workload("t", 2, 2, 2, 16, 4096, 16, dtype="bf16", k_offset_std=4.0)
    _, k, v = dense_inputs(w, 0)
    kf = k.float()
    # the offset is identical for every batch entry and token: the per-(b, h, c) means over
    # tokens of the two batch entries agree up to the unit-variance noise (~1/sqrt(4096))
    m = kf.mean(dim=2)                                   # [B, H, d]
    assert (m[0] - m[1]).abs().max() < 0.1
    assert m.abs().mean() > 1.0                          # a std-4 offset dominates the noise
    # no offset on V (v_offset_std = 0): per-channel means stay near 0
    assert v.float().mean(dim=2).abs().max() < 0.1
    assert k.dtype == torch.bfloat16


def test_nhd_is_a_pure_layout():
    w_h = Workload("t", 1, 3, 3, 40, 40, 8)
    w_n = Workload("t", 1, 3, 3, 40, 40, 8, layout="NHD")
    for a, b in zip(dense_inputs(w_h, 5), dense_inputs(w_n, 5)):
        assert torch.equal(a.transpose(1, 2), b)
        assert (to_hnd_f32(a, "HND") == to_hnd_f32(b, "NHD")).all()


def test_varlen_lengths_and_packing():
    w = WORKLOADS["varlen16"]
    lens = varlen_lengths(w, 0)
    assert len(lens) == 16 and all(128 <= n <= 8192 for n in lens)
    assert lens == varlen_lengths(w, 0)
    small = Workload("v", 3, 4, 2, 0, 0, 16, varlen=True, n_seqs=3)
    q, k, v, cu_q, cu_k, got = varlen_inputs(small, 1, [5, 0, 7])
    assert got == [5, 0, 7]
    assert cu_q.tolist() == [0, 5, 5, 12] and torch.equal(cu_q, cu_k) and cu_q.dtype == torch.int32
    assert q.shape == (12, 4, 16) and k.shape == (12, 2, 16) and v.shape == (12, 2, 16)


def test_operation_counts():
    w = WORKLOADS["sdpa4k"]
    assert w.ops() == 4.0 * 2 * 8 * 4096 * 4096 * 128
    c = WORKLOADS["gqa_causal8k"]
    assert c.ops() == 4.0 * 1 * 32 * 8192 * 8192 * 128 / 2
    vl = Workload("v", 2, 4, 4, 0, 0, 64, varlen=True, n_seqs=2)
    assert vl.ops([3, 5]) == 4.0 * 4 * (9 + 25) * 64
