"""Replica bookkeeping for runs on several GPUs of one node.

The hot path has no exchange step: sequences are independent, so N GPUs run N independent
replicas of the step (one process per GPU, launched by torchrun) and no collective touches
the data path.  The only collectives are for measurement: a barrier before and after the
timed region and the maximum of the ranks' elapsed times, from which the job's aggregate
throughput is computed.  Works with any torch.distributed backend (nccl on GPUs, gloo on CPU).
"""

from __future__ import annotations

import os


def rank_info():
    """(rank, world_size, local_rank) from the torchrun environment; (0, 1, 0) if absent."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest `value` over all ranks (the slowest replica sets the job's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world_size, max_seconds):
    """Whole-job throughput: every rank processed `units_per_rank` in at most `max_seconds`."""
    if max_seconds <= 0:
        raise ValueError("elapsed time must be positive")
    return world_size * units_per_rank / max_seconds
