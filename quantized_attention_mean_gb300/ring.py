"""Ring (context-parallel) attention over a process group, composed from ``sage_attn`` and
``merge_partials``.

The forward returns the log-sum-exp of every query row "for Ring Attention and similar"
schemes (pwwt.cn "SageAttention deployment pitfalls guide" §4.1): the keys are split into
chunks that are attended to separately and the partial outputs are combined through their
LSE. Here each rank of the group holds one contiguous shard of a long sequence (its queries
and its keys / values, shard r covering token positions [r N, (r + 1) N) of the sequence);
the K / V shards travel around the ring, one hop per step, while every rank attends its own
queries to the shard it currently holds:

    step s: rank r holds K / V shard (r - s) mod W; it sends that shard to rank r + 1 and
            receives the next one from rank r - 1 (both into its own buffers) while it
            computes the partial attention of its queries to the shard it holds.

After W steps every rank has seen every shard, and ``merge_partials`` combines its partial
results. With ``is_causal`` a query shard attends fully to earlier key shards, causally
(top-left, positions aligned) to its own, and skips later ones. Each partial uses the
method's per-shard smoothing and quantisation; the LSE of each partial includes the smooth_k
correction, so the merge is exact for the partials given.

Communication uses ``torch.distributed`` point-to-point sends and receives (NCCL between
GPUs, gloo on the CPU); the data path adds no collective.
"""

import torch
import torch.distributed as dist

__all__ = ["ring_chunk", "chunk_mode", "ring_attention"]


def ring_chunk(rank, world, step):
    """The K / V shard rank `rank` holds at ring step `step` (0 <= step < world)."""
    return (rank - step) % world


def chunk_mode(q_shard, k_shard, is_causal):
    """How query shard `q_shard` attends to key shard `k_shard`: "full", "causal" (the
    diagonal shard: key j visible to query i iff j <= i) or "none"."""
    if not is_causal or k_shard < q_shard:
        return "full"
    return "causal" if k_shard == q_shard else "none"


def _sage_attend(q, k, v, causal, tensor_layout, **kw):
    from . import sage_attn
    return sage_attn(q, k, v, tensor_layout=tensor_layout, is_causal=causal, return_lse=True, **kw)


def _sage_merge(outs, lses, tensor_layout):
    from . import merge_partials
    return merge_partials(outs, lses, tensor_layout=tensor_layout)


def ring_attention(q, k, v, *, group=None, is_causal=False, tensor_layout="HND", attend=None,
                   merge=None, **sage_kwargs):
    """Ring attention of this rank's query shard over every rank's K / V shard.

    q: this rank's queries, k / v: this rank's keys / values ([B, H, N, d] for HND,
    [B, N, H, d] for NHD); every rank's k / v shards must have the same shape and dtype.
    Returns (out, lse) for this rank's queries. `attend(q, k, v, causal, tensor_layout,
    **sage_kwargs) -> (out, lse)` and `merge(outs, lses, tensor_layout) -> (out, lse)` default
    to ``sage_attn`` (with return_lse) and ``merge_partials`` on the GPU; another pair can be
    passed to run the same schedule on other tensors. Extra keyword arguments go to `attend`.
    """
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    attend = _sage_attend if attend is None else attend
    merge = _sage_merge if merge is None else merge
    peer = (lambda r: r) if group is None else (lambda r: dist.get_global_rank(group, r))
    send_to, recv_from = peer((rank + 1) % world), peer((rank - 1) % world)
    # the caller's shard is only read and sent; shards arriving from the ring alternate
    # between two receive buffers (the one received two steps ago has been sent on by then)
    cur_k, cur_v = k.contiguous(), v.contiguous()
    recv = [(torch.empty_like(cur_k), torch.empty_like(cur_v)) for _ in range(min(2, world - 1))]
    outs, lses = [], []
    for step in range(world):
        reqs = []
        if step + 1 < world:
            nxt_k, nxt_v = recv[step % 2]
            ops = [dist.P2POp(dist.isend, cur_k, send_to, group),
                   dist.P2POp(dist.isend, cur_v, send_to, group),
                   dist.P2POp(dist.irecv, nxt_k, recv_from, group),
                   dist.P2POp(dist.irecv, nxt_v, recv_from, group)]
            reqs = dist.batch_isend_irecv(ops)
        mode = chunk_mode(rank, ring_chunk(rank, world, step), is_causal)
        if mode != "none":
            o, l = attend(q, cur_k, cur_v, mode == "causal", tensor_layout, **sage_kwargs)
            outs.append(o)
            lses.append(l)
        for r in reqs:
            r.wait()
        if step + 1 < world:
            cur_k, cur_v = recv[step % 2]
    return merge(outs, lses, tensor_layout)
