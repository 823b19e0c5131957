"""Process-rank plumbing for one replica per GPU.

The fused path has no exchange step ("DirectKV: ... zero-copy KV cache", the
multi-GPU discussion of the problem statement: each GPU reads its own pinned
cache slice over its own host link), so N GPUs run N independent replicas:
every rank serves its own sequences and the only collectives are on the
timing path (a barrier around the timed region and a max over ranks of the
elapsed time).  This module holds that host logic so it can be exercised on
CPU ranks (gloo) as well as under torchrun on GPUs (nccl).
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class Ranks:
    world: int
    rank: int
    local: int

    @staticmethod
    def from_env(env=None) -> "Ranks":
        """WORLD_SIZE / RANK / LOCAL_RANK as torchrun exports them (1 / 0 / 0 if unset)."""
        env = os.environ if env is None else env
        world = int(env.get("WORLD_SIZE", "1"))
        rank = int(env.get("RANK", "0"))
        local = int(env.get("LOCAL_RANK", str(rank)))
        if world < 1 or not 0 <= rank < world or local < 0:
            raise ValueError(f"bad rank environment: world={world} rank={rank} local={local}")
        return Ranks(world, rank, local)


def shard(n_units: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous block [lo, hi) of n_units owned by `rank`.

    The first n_units % world ranks take one unit more, so block sizes differ
    by at most one and the blocks tile [0, n_units) in rank order.
    """
    if world < 1 or not 0 <= rank < world or n_units < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n_units, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def _active(dist) -> bool:
    return dist is not None and dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def barrier(dist=None) -> None:
    if _active(dist):
        dist.barrier()


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest `value` any rank holds (the slowest rank's time); the value itself alone."""
    if not _active(dist):
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    if seconds_max <= 0:
        raise ValueError("elapsed time must be positive")
    return units_per_rank * world / seconds_max
