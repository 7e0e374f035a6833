"""Data-parallel replicas of the sampler step: one process per GPU, each serving its own
canvases (independent requests), no collective on the data path.

Host-side logic only: which workload a rank serves, and how per-rank timings become
one whole-job number (the slowest rank sets the time; every rank's positions count).
"""
from __future__ import annotations

from . import inputs

SEED_STRIDE = 1000


def rank_workload(base: "inputs.Workload", rank: int) -> "inputs.Workload":
    """The canvases rank `rank` serves: the same shapes, its own seeded draw."""
    return base.with_(seed=base.seed + SEED_STRIDE * rank)


def max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over all ranks of the default process group
    (the input unchanged when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(rows_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Positions per second of the whole job: every rank's rows over the slowest rank's time."""
    return world * rows_per_rank * steps / (max_ms * 1e-3)
