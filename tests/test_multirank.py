"""bench.py's multi-rank logic on CPU with two gloo ranks: barrier, max-over-ranks timing,
and whole-job (weak-scaling) throughput = all ranks' operations over the slowest rank."""

import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    bench.init_dist(ws, local, "gloo")
    bench.barrier(ws)
    my_seconds = 1.0 + rank          # rank 1 is the slow one
    mx = bench.max_over_ranks(my_seconds, ws)
    value = bench.aggregate(1e12, 10, mx, ws)
    q.put((rank, ws, mx, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ws, mx, value in res:
        assert ws == 2
        assert mx == 2.0                           # max over ranks
        assert abs(value - 1e12 * 10 * 2 / 2.0 / 1e12) < 1e-9   # 10 TOPS whole-job


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate(2e12, 5, 2.0, 1) == 5.0
