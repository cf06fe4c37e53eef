"""Host-side helpers for running the library on several GPUs, one process each.

Rows are independent, so a batch splits across ranks by rows with no exchange
of data: rank r takes the contiguous block ``shard_rows(rows, r, world)`` and
calls the library on it.  The only cross-rank step is bookkeeping: a barrier
and the maximum of the per-rank times (``max_over_ranks``), which the
benchmark uses to report whole-job throughput.  Works with any
torch.distributed backend (NCCL between GPUs, gloo on CPU).
"""
from __future__ import annotations


def shard_rows(rows: int, rank: int, world: int) -> tuple[int, int]:
    """[begin, end) of rank's block of rows; blocks differ in size by at most one."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("need rows >= 0 and 0 <= rank < world")
    base, extra = divmod(rows, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of `value` over all ranks of the default process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units processed by all ranks per second of the slowest rank."""
    if max_seconds <= 0:
        raise ValueError("time must be positive")
    return units_per_rank * world / max_seconds
