"""Host-side bookkeeping for a run on N GPUs of one node.

The hot path shards into independent replicas: the linears and the
verification of one batch need nothing from another GPU, so N GPUs run N
copies of the step with no exchange on the data path.  The only multi-rank
steps are on the host: a barrier on each side of the timed region, the maximum
over ranks of the measured times, and the whole-job rate (the units all ranks
processed over the slowest rank's time).  torch.distributed carries them:
NCCL on GPUs, gloo in the CPU tests.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def world_rank_local():
    """(WORLD_SIZE, RANK, LOCAL_RANK) from the launcher's environment, 1/0/0 alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def barrier(world: int) -> None:
    if world > 1:
        dist.barrier()


def max_over_ranks(values, world: int, device) -> list:
    """Element-wise maximum over ranks of a list of floats (times)."""
    if world == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world: int, units_per_rank: float, seconds: float) -> float:
    """Units all ranks processed (each the same amount: weak scaling) per
    second of the slowest rank."""
    return world * units_per_rank / seconds
