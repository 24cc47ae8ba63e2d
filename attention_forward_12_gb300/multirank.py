"""Host logic of running the forward on several GPUs, one process per GPU.

The (batch, head) problems of the forward are independent, so ranks share no
data: each rank runs its own problems on its own GPU and the only
cross-rank traffic is the benchmark's timing reduction.  Nothing here
touches the data path.
"""
from __future__ import annotations


def rank_seed(seed: int, rank: int) -> int:
    """Seed of rank `rank`'s independent problems (rank 0 keeps `seed`)."""
    return int(seed) + 7919 * int(rank)


def shard_heads(BH: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [lo, hi) range of the B*H heads owned by `rank` when one
    problem is split across ranks; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or BH < 0:
        raise ValueError("bad rank / world / BH")
    base, extra = divmod(BH, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """Maximum of `value` over all ranks of the default process group (the
    slowest rank sets the time of a step); identity without a group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank: float, world: int, step_ms: float) -> float:
    """Whole-job throughput: the FLOP of every rank over the slowest rank's time."""
    return world * flops_per_rank / (step_ms * 1e-3) / 1e12
