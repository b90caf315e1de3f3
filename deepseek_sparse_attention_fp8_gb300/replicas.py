"""Aggregation of per-rank timings when several GPUs run independent replicas.

The DSA step has no exchange between query tokens, so N GPUs run N replicas
of the same step with no collective on the data path. Only the benchmark's
bookkeeping talks across ranks: the slowest rank's time bounds the job, and
the tokens of all ranks add up.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def aggregate(ms_local: float, tokens_local: int, device=None):
    """Returns (max ms over ranks, total tokens over ranks, tokens/s of the job)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms_local, tokens_local, tokens_local / (ms_local / 1e3)
    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    n = torch.tensor([float(tokens_local)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    ms, tokens = float(t.item()), int(round(n.item()))
    return ms, tokens, tokens / (ms / 1e3)
