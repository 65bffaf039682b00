"""Data-parallel replicas: requests are independent through drafting,
context injection and verification, so N GPUs each run their own copy of the
drafter on a disjoint slice of the requests.  There is no collective on the
data path; the only cross-rank traffic is host-side bookkeeping (a barrier and
the maximum of the per-rank step times that turns per-rank work into a
whole-job throughput)."""

import torch


def partition(n_requests, world, rank):
    """Contiguous, balanced slice [start, stop) of request indices for `rank`."""
    if world < 1 or not 0 <= rank < world or n_requests < 0:
        raise ValueError("bad partition arguments")
    base, extra = divmod(n_requests, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(x, device=None):
    """Maximum of a scalar over all ranks of the default process group
    (identity when torch.distributed is not initialised)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, seconds_per_rank):
    """Whole-job units/s: all units processed divided by the slowest rank's time."""
    return float(sum(units_per_rank)) / max(seconds_per_rank)
