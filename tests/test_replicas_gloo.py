"""World-size-2 gloo run (CPU) of the multi-GPU bookkeeping: each rank runs its
own replica; the job time is the slowest rank's and the work is the sum."""

import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

from dual_mode_canvas_gb300 import replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 if rank == 0 else 25.0
        units = 100.0 * (rank + 1)
        replicas.barrier()
        got = replicas.aggregate(ms, units)
        tp = replicas.throughput(ms, units)
        q.put((rank, got, tp, replicas.world()))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (ms, units), tp, (n, r) in res:
        assert n == 2 and r == rank
        assert ms == 25.0 and units == 300.0
        assert abs(tp - 300.0 / 0.025) < 1e-6


def test_single_process_is_identity():
    assert replicas.aggregate(3.0, 7.0) == (3.0, 7.0)
    assert replicas.world() == (1, 0)
