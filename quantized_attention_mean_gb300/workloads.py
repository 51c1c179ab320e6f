"""Seeded synthetic inputs shaped like the workloads the method is used on.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic. Both the CUDA path's tests/benchmark and the CPU oracle receive the same
tensors from it.

Recipe: one CPU generator per tensor, seeded with `seed`, drawn in fp32 in the order
Q, K, (K per-channel offset), V, (V per-channel offset); "N(0, s)" means standard
deviation s; a per-channel offset has shape [H_kv, d] and is shared by every batch entry
and token (the outlier structure smoothing is meant for); values are then rounded to
fp16/bf16 (round-to-nearest-even, torch's cast) and laid out HND [B, H, N, d] or NHD
[B, N, H, d]. Varlen batches draw their lengths uniformly from [128, 8192] with the
same seed and pack tokens as [T, H, d].
"""

from dataclasses import dataclass, field

import torch

GRAN = {"per_block": 0, "per_warp": 1, "per_thread": 2}
ACC = {"fp32": 0, "fp16+fp32": 1, "fp32+fp32": 2, "fp16": 3}
DTYPE = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    dtype: str = "fp16"
    layout: str = "HND"
    is_causal: bool = False
    gran: str = "per_warp"
    accum: str = "fp32"
    smooth_k: bool = True
    smooth_v: bool = False
    return_lse: bool = False
    k_offset_std: float = 0.0
    v_offset_std: float = 0.0
    varlen: bool = False
    n_seqs: int = 0
    len_range: tuple = (128, 8192)
    extra: dict = field(default_factory=dict)

    def ops(self, seqlens=None):
        """4·B·H·Nq·Nk·d, halved when causal; summed per sequence for varlen."""
        if self.varlen:
            tot = sum(int(n) * int(n) for n in seqlens)
            return 4.0 * self.Hq * tot * self.d / (2.0 if self.is_causal else 1.0)
        return 4.0 * self.B * self.Hq * self.Nq * self.Nk * self.d / (2.0 if self.is_causal else 1.0)


# The five workloads the method is measured on (tiny check, standard 4K self-attention,
# a causal decoder with grouped KV heads, a video-diffusion-transformer-shaped long
# sequence with biased K and V, and a ragged serving batch).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 2, 256, 256, 64, gran="per_block", accum="fp32"),
    "sdpa4k": Workload("sdpa4k", 2, 8, 8, 4096, 4096, 128, gran="per_warp", accum="fp16+fp32"),
    "gqa_causal8k": Workload("gqa_causal8k", 1, 32, 8, 8192, 8192, 128, dtype="bf16",
                             layout="NHD", is_causal=True, gran="per_thread", accum="fp32",
                             return_lse=True, k_offset_std=3.0),
    "dit17776": Workload("dit17776", 2, 48, 48, 17776, 17776, 64, dtype="bf16", gran="per_warp",
                         accum="fp16+fp32", smooth_v=True, k_offset_std=4.0, v_offset_std=2.0),
    # the 4K self-attention shape on the FP16 P·V variant
    "sdpa4k_pv16": Workload("sdpa4k_pv16", 2, 8, 8, 4096, 4096, 128, gran="per_warp",
                            accum="fp16+fp32", extra={"pv": "fp16"}),
    # half the heads of the DiT shape at batch 1 (same per-CTA work): a profiling case whose
    # attention launch is short enough for a multi-pass ncu capture
    "dit17776_h24": Workload("dit17776_h24", 1, 24, 24, 17776, 17776, 64, dtype="bf16",
                             gran="per_warp", accum="fp16+fp32", smooth_v=True, k_offset_std=4.0,
                             v_offset_std=2.0),
    # the DiT shape and the 4K self-attention shape on the FP4 microscaled variant
    "dit17776_fp4": Workload("dit17776_fp4", 2, 48, 48, 17776, 17776, 64, dtype="bf16",
                             gran="per_warp", accum="fp16+fp32", smooth_v=True, k_offset_std=4.0,
                             v_offset_std=2.0, extra={"pv": "fp4"}),
    "sdpa4k_fp4": Workload("sdpa4k_fp4", 2, 8, 8, 4096, 4096, 128, gran="per_warp",
                           accum="fp16+fp32", extra={"pv": "fp4"}),
    # the FP4 variant on half the DiT heads at batch 1 (a profiling case, as dit17776_h24)
    "dit17776_fp4_h24": Workload("dit17776_fp4_h24", 1, 24, 24, 17776, 17776, 64, dtype="bf16",
                                 gran="per_warp", accum="fp16+fp32", smooth_v=True, k_offset_std=4.0,
                                 v_offset_std=2.0, extra={"pv": "fp4"}),
    "varlen16": Workload("varlen16", 16, 32, 32, 0, 0, 128, gran="per_warp", accum="fp32",
                         varlen=True, n_seqs=16),
}


def _draw(shape, std, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * std


def _gen(seed):
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return g


def dense_inputs(w: Workload, seed=0):
    """CPU tensors q, k, v in w.dtype and w.layout (HND [B,H,N,d] / NHD [B,N,H,d])."""
    dt = DTYPE[w.dtype]
    q = _draw((w.B, w.Hq, w.Nq, w.d), 1.0, _gen(seed))
    k = _draw((w.B, w.Hkv, w.Nk, w.d), 1.0, _gen(seed + 1))
    if w.k_offset_std:
        k = k + _draw((w.Hkv, w.d), w.k_offset_std, _gen(seed + 2))[None, :, None, :]
    v = _draw((w.B, w.Hkv, w.Nk, w.d), 1.0, _gen(seed + 3))
    if w.v_offset_std:
        v = v + _draw((w.Hkv, w.d), w.v_offset_std, _gen(seed + 4))[None, :, None, :]
    q, k, v = (t.to(dt) for t in (q, k, v))
    if w.layout == "NHD":
        q, k, v = (t.transpose(1, 2).contiguous() for t in (q, k, v))
    return q, k, v


def varlen_lengths(w: Workload, seed=0):
    lo, hi = w.len_range
    return torch.randint(lo, hi + 1, (w.n_seqs,), generator=_gen(seed)).tolist()


def varlen_inputs(w: Workload, seed=0, lengths=None):
    """Packed CPU tensors q [Tq,Hq,d], k/v [Tk,Hkv,d] and int32 cu_seqlens (q == k)."""
    lengths = varlen_lengths(w, seed) if lengths is None else list(lengths)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    t = int(cu[-1])
    dt = DTYPE[w.dtype]
    q = _draw((t, w.Hq, w.d), 1.0, _gen(seed + 11)).to(dt)
    k = _draw((t, w.Hkv, w.d), 1.0, _gen(seed + 12))
    if w.k_offset_std:
        k = k + _draw((w.Hkv, w.d), w.k_offset_std, _gen(seed + 13))[None]
    v = _draw((t, w.Hkv, w.d), 1.0, _gen(seed + 14))
    if w.v_offset_std:
        v = v + _draw((w.Hkv, w.d), w.v_offset_std, _gen(seed + 15))[None]
    return q, k.to(dt), v.to(dt), cu, cu.clone(), lengths


def to_hnd_f32(t, layout):
    """Exact fp16/bf16 -> fp32 copy in [B, H, N, d] order (layout is pure indexing)."""
    t = t.float()
    return (t.transpose(1, 2) if layout == "NHD" else t).contiguous().numpy()
