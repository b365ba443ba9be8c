"""Data-parallel replicas: one process per GPU, each with its own sequences.

The decode path has no exchange step between sequences: every (layer,
sequence, KV head) reads only its own pages.  N GPUs therefore run N
independent replicas of the workload (weak scaling), each drawing its own
sequences from a rank-offset seed, and the only collectives are the host-side
barrier around each timed region and the max of the region's time over ranks.
"""
from __future__ import annotations

import dataclasses
import os

import torch
import torch.distributed as dist


@dataclasses.dataclass(frozen=True)
class Ranks:
    world: int
    rank: int
    local: int


def from_env() -> Ranks:
    """World size, rank and local rank as torchrun exports them (1, 0, 0 alone)."""
    return Ranks(int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
                 int(os.environ.get("LOCAL_RANK", "0")))


def shard(workload, rank: int):
    """This rank's replica: the same shapes, its own sequences (seed offset by rank)."""
    return workload if rank == 0 else workload.scaled(seed=workload.seed + 1000003 * rank)


def barrier(r: Ranks) -> None:
    if r.world > 1:
        dist.barrier()


def max_over_ranks(r: Ranks, seconds: float, device) -> float:
    """The slowest rank's time for a region every rank timed."""
    if r.world == 1:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(r: Ranks, units_per_rank: int, seconds_max: float) -> float:
    """Units all ranks processed per second of the slowest rank."""
    return r.world * units_per_rank / seconds_max
