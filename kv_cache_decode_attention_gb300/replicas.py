"""Host-side bookkeeping for running the decode path on several GPUs of one node.

Decode attention needs no exchange between sequences: every (sequence, layer)
decode step is an independent unit.  Across GPUs the library therefore runs
independent replicas (weak scaling: each rank owns its own batch of
sequences on its own GPU) and only the timing is combined: a barrier on each
side of the timed region and the maximum elapsed time over ranks.  Nothing
on the data path crosses GPUs.
"""

from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class RankInfo:
    rank: int
    world: int
    local_rank: int

    @property
    def is_root(self) -> bool:
        return self.rank == 0


def rank_info(env=None) -> RankInfo:
    """Rank, world size and local rank from the torchrun environment (1 rank if unset)."""
    env = os.environ if env is None else env
    world = int(env.get("WORLD_SIZE", "1"))
    rank = int(env.get("RANK", "0"))
    local = int(env.get("LOCAL_RANK", str(rank)))
    if world < 1 or not (0 <= rank < world):
        raise ValueError("bad rank %d of world %d" % (rank, world))
    return RankInfo(rank, world, local)


def sequence_seed(base_seed: int, rank: int) -> int:
    """Seed of a rank's replica: distinct per rank so replicas hold different
    sequences, identical on every run."""
    return base_seed + 1_000_003 * rank


def max_over_ranks(value: float, group=None) -> float:
    """The largest `value` over all ranks (plain float on one rank).  Uses the
    process group's backend (nccl on GPUs, gloo on CPU)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def barrier(group=None) -> None:
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier(group=group)


def whole_job_rate(units_per_rank: float, elapsed_s_max: float, world: int) -> float:
    """Throughput of the whole job: every rank processed `units_per_rank` in at
    most `elapsed_s_max` seconds."""
    if elapsed_s_max <= 0:
        raise ValueError("elapsed time must be positive")
    return units_per_rank * world / elapsed_s_max
