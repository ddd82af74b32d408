"""Multi-GPU bookkeeping for ``bench.py --gpus N``.

The attention path shards without any exchange: sequences, KV heads and query
tiles are independent, so N GPUs run N independent replicas of the workload
(weak scaling) and nothing crosses ranks on the data path.  Only the timing
summary does: the job time is the slowest rank's time and the work is the sum
over ranks.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def world() -> tuple[int, int]:
    if dist.is_available() and dist.is_initialized():
        return dist.get_world_size(), dist.get_rank()
    return 1, 0


def aggregate(local_ms: float, local_units: float, device="cpu") -> tuple[float, float]:
    """(max over ranks of ``local_ms``, sum over ranks of ``local_units``)."""
    n, _ = world()
    if n == 1:
        return float(local_ms), float(local_units)
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    u = torch.tensor([local_units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def throughput(local_ms: float, local_units: float, device="cpu") -> float:
    """Whole-job units per second: all ranks' units over the slowest rank's time."""
    ms, units = aggregate(local_ms, local_units, device)
    return units / (ms * 1e-3)


def barrier():
    n, _ = world()
    if n > 1:
        dist.barrier()
