"""Ring attention's exchange schedule (quantized_attention_mean_gb300.ring) with gloo ranks on
the CPU: every rank must end with the merge of its queries' partial attention over every K / V
shard (fully to earlier shards, causally to its own, not at all to later ones when causal).
The ranks run the library's ring schedule with the oracle's attention and merge passed in as
the per-shard compute; the expected result merges the same per-shard oracle partials computed
directly from all shards, so the test checks the sends, receives, buffer rotation and shard
bookkeeping. The ranks' output is also checked against float64 attention over the whole
sequence (cosine). On the GPU the same schedule runs sage_attn and merge_partials over NCCL
(not run here: one GPU)."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs(world, n, seed=0):
    g = torch.Generator().manual_seed(seed)
    shape = (1, 2, world * n, 32)
    q = torch.randn(shape, generator=g).half().float()
    k = (torch.randn(shape, generator=g) + torch.randn((1, 2, 1, 32), generator=g) * 2).half().float()
    v = torch.randn(shape, generator=g).half().float()
    return q, k, v


def _oracle_attend(q, k, v, causal, tensor_layout, **kw):
    from oracle.attention import sage_attention
    r = sage_attention(q.numpy(), k.numpy(), v.numpy(), is_causal=causal, **kw)
    return torch.from_numpy(r["o"]), torch.from_numpy(r["lse"])


def _oracle_merge(outs, lses, tensor_layout):
    from oracle.merge import merge_partials
    o, l = merge_partials([x.numpy() for x in outs], [x.numpy() for x in lses])
    return torch.from_numpy(o), torch.from_numpy(l)


def _worker(rank, world, port, n, causal, q_out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from quantized_attention_mean_gb300.ring import ring_attention
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v = _inputs(world, n)
    sl = slice(rank * n, (rank + 1) * n)
    o, l = ring_attention(q[:, :, sl], k[:, :, sl].contiguous(), v[:, :, sl].contiguous(),
                          is_causal=causal, attend=_oracle_attend, merge=_oracle_merge,
                          sm_scale=0.2, smooth_v=True)
    q_out.put((rank, o.numpy(), l.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,causal", [(2, False), (2, True), (3, True)])
def test_ring_schedule_with_gloo_ranks(world, causal):
    sys.path.insert(0, ROOT)
    from oracle.attention import attention_fp64
    from quantized_attention_mean_gb300.ring import chunk_mode
    n = 40
    ctx = mp.get_context("spawn")
    qq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, causal, qq)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, o, l = qq.get(timeout=300)
        got[r] = (o, l)
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    q, k, v = _inputs(world, n)
    for r in range(world):
        sq = slice(r * n, (r + 1) * n)
        outs, lses = [], []
        for c in range(world):
            mode = chunk_mode(r, c, causal)
            if mode == "none":
                continue
            sk = slice(c * n, (c + 1) * n)
            o, l = _oracle_attend(q[:, :, sq], k[:, :, sk], v[:, :, sk], mode == "causal", "HND",
                                  sm_scale=0.2, smooth_v=True)
            outs.append(o)
            lses.append(l)
        want_o, want_l = _oracle_merge(outs, lses, "HND")
        np.testing.assert_allclose(got[r][0], want_o.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(got[r][1], want_l.numpy(), rtol=0, atol=1e-12)
        # the composition is attention over the whole (causal) sequence, up to quantisation
        for h in range(2):
            rows = np.arange(r * n, (r + 1) * n)
            of, lf = attention_fp64(q[0, h].numpy(), k[0, h].numpy(), v[0, h].numpy(), 0.2, causal, rows=rows)
            a, b = got[r][0][0, h].ravel(), of.ravel()
            assert a @ b / (np.linalg.norm(a) * np.linalg.norm(b)) > 0.99
            assert np.abs(got[r][1][0, h] - lf).max() < 0.05


def test_ring_bookkeeping():
    from quantized_attention_mean_gb300.ring import chunk_mode, ring_chunk
    # every rank sees every shard exactly once over the steps
    for world in (1, 2, 5):
        for rank in range(world):
            assert sorted(ring_chunk(rank, world, s) for s in range(world)) == list(range(world))
    assert chunk_mode(2, 1, True) == "full" and chunk_mode(2, 2, True) == "causal"
    assert chunk_mode(2, 3, True) == "none" and chunk_mode(2, 3, False) == "full"


@pytest.mark.gpu
def test_ring_default_path_on_one_gpu():
    # a one-rank group runs the default compute (sage_attn with return_lse, merge_partials)
    # with no exchange: the merge of the single partial is the partial itself
    import torch.distributed as dist
    import quantized_attention_mean_gb300 as qa
    from quantized_attention_mean_gb300.ring import ring_attention
    dev = torch.device("cuda:0")
    q, k, v = (t.half().to(dev) for t in _inputs(1, 300, seed=3))
    store = dist.HashStore()
    group_init = not dist.is_initialized()
    if group_init:
        dist.init_process_group("gloo", store=store, rank=0, world_size=1)
    try:
        o, l = ring_attention(q, k, v, is_causal=True, smooth_v=True)
        ref_o, ref_l = qa.sage_attn(q, k, v, is_causal=True, return_lse=True, smooth_v=True)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o)
        assert torch.allclose(l, ref_l, rtol=0, atol=1e-6)
    finally:
        if group_init:
            dist.destroy_process_group()
