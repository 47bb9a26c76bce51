"""Host logic of a multi-process run: one process per GPU, each an independent
replica of the whole call on its own batch (the attention call shards over
documents and heads with no exchange step, so no collective sits on the data
path).  Only the timing is shared: every rank reports its timed total, the
slowest one counts, and the whole-job throughput is the work of all ranks
over that time.

Backend-agnostic (NCCL with CUDA tensors on a GPU machine, gloo with CPU tensors
in tests)."""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class RankEnv:
    world: int
    rank: int
    local: int


def rank_env(environ=None) -> RankEnv:
    """WORLD_SIZE / RANK / LOCAL_RANK as set by torch.distributed.run (1 / 0 / 0 without it)."""
    e = os.environ if environ is None else environ
    world = int(e.get("WORLD_SIZE", "1"))
    rank = int(e.get("RANK", "0"))
    local = int(e.get("LOCAL_RANK", str(rank)))
    if world < 1 or not 0 <= rank < world or local < 0:
        raise ValueError(f"inconsistent rank environment: world {world}, rank {rank}, local {local}")
    return RankEnv(world, rank, local)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest of every rank's ``value`` (the value itself without a process group)."""
    if dist is None or not dist.is_initialized():
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_step: float, steps: int, slowest_total_ms: float) -> float:
    """Units per second of the whole job: every rank processed ``steps`` steps
    of ``units_per_step`` units, and the job took the slowest rank's time."""
    if slowest_total_ms <= 0 or steps <= 0:
        raise ValueError("a timed run needs steps > 0 and a positive time")
    return world * units_per_step * steps / (slowest_total_ms * 1e-3)
