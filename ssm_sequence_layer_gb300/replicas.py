"""Host-side logic of multi-GPU runs.

The recurrence of each (batch, head) sequence is independent of every other one, so the
path has no exchange step: N GPUs either run N independent replicas of a workload (the
benchmark's weak scaling) or split the B*H sequences between them.  Neither needs a
collective on the data path; torch.distributed is used only for a barrier before and after
a timed region and for taking the maximum time over ranks.
"""
from __future__ import annotations


def shard_sequences(B: int, H: int, world: int, rank: int):
    """Contiguous share of the B*H (batch, head) sequences for `rank` of `world`.

    Returns (start, stop) in the flattened b*H + h order; the shares cover every sequence
    exactly once and differ in size by at most one.
    """
    if world < 1 or not (0 <= rank < world):
        raise ValueError("need 0 <= rank < world")
    units = B * H
    base, extra = divmod(units, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
