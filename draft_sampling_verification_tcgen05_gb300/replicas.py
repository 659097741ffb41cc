"""Replica orchestration on one node: one process per GPU, each serving its own requests.

The draft step, the verification and the admission pool of a request depend on no
other request ("DSpark implementation and evaluation" §3 keeps the Markov head
replicated rather than tensor-parallel for this reason), so N GPUs run N replicas
with replicated weights and no data-path collective.  Ranks meet only to agree on
the timing of a step (the slowest rank sets the job's pace).  This module holds that
host logic; it imports no CUDA code, so it runs (and is tested) on CPU ranks too.
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class RankInfo:
    rank: int
    world: int
    local_rank: int


def rank_info(env=None) -> RankInfo:
    """RANK / WORLD_SIZE / LOCAL_RANK as set by torch.distributed.run (defaults: one process)."""
    env = os.environ if env is None else env
    rank = int(env.get("RANK", "0"))
    world = int(env.get("WORLD_SIZE", "1"))
    local = int(env.get("LOCAL_RANK", str(rank)))
    if world < 1 or not 0 <= rank < world or local < 0:
        raise ValueError(f"inconsistent rank environment: RANK={rank} WORLD_SIZE={world} LOCAL_RANK={local}")
    return RankInfo(rank, world, local)


def shard_range(n_global: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous share [lo, hi) of n_global requests for `rank`; shares differ by at most one."""
    if n_global < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n_global, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def replica_seed(seed: int, rank: int) -> int:
    """Philox seed of a replica: the replicas' requests draw independent streams (the rank
    goes into the upper half of the 64-bit key, which the single-GPU seeds leave at 0)."""
    return (int(seed) & 0xFFFFFFFF) | (int(rank) << 32)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (every rank gets it); `value` itself without a group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job rate: the units all ranks processed per second of the slowest rank's time."""
    if max_ms <= 0:
        raise ValueError("time must be positive")
    return world * units_per_rank / (max_ms / 1e3)
