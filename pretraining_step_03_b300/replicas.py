"""Data-parallel replicas of the training step: one process per GPU, no collective
on the data path.

Every rank trains its own model copy on its own synthetic rows (the step has no
exchange other than the gradient all-reduce of data parallelism, which a set of
independent replicas does not perform).  Only the measurement is combined: the
timed region is bracketed by barriers, the job's step time is the slowest rank's,
and the whole-job rate counts every rank's tokens.  The host-side logic lives here
so it can be exercised with the gloo backend on CPU.
"""

import os


def rank_env():
    """(rank, world_size, local_rank) from the launcher's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def data_seed(rank, base=1):
    """Seed of a rank's synthetic token rows (distinct per rank)."""
    return base + rank


def max_over_ranks(value, dist=None, device=None):
    """The maximum of a per-rank scalar over all ranks (the value itself without a group)."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, tokens_per_step, seconds_per_step):
    """Whole-job tokens per second: every rank's tokens over the slowest rank's step time."""
    return world * tokens_per_step / seconds_per_step
