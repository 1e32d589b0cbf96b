"""Running the hot path on several GPUs.

Every (request, layer) unit is independent (gentlecold.top "HiSparse 深度解析"
§3.3, last paragraph: each layer of each request manages its own cache), so
the work splits by request with no exchange between GPUs: each rank owns its
requests' hot buffers, metadata and host-pool rows.  The only cross-rank
operations are outside the hot path: a barrier around timed regions and a MAX
reduction of the elapsed time.
"""


def shard_requests(total_requests, world_size, rank):
    """Contiguous block of requests for `rank`: (first request, count)."""
    if world_size < 1 or not 0 <= rank < world_size or total_requests < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(total_requests, world_size)
    count = base + (1 if rank < extra else 0)
    first = rank * base + min(rank, extra)
    return first, count


def replica_seed(seed, rank):
    """Seed of rank `rank`'s own replica of a workload (weak scaling)."""
    return seed + 1000 * rank


def max_over_ranks(value, dist=None, device=None):
    """MAX of a float over all ranks (identity without a process group)."""
    if dist is None or not dist.is_available() or not dist.is_initialized():
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, seconds_max, world_size):
    """Whole-job rate: units every rank processed over the slowest rank's time."""
    if seconds_max <= 0:
        raise ValueError("elapsed time must be positive")
    return units_per_rank * world_size / seconds_max
