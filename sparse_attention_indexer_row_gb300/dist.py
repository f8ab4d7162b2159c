"""Host-side helpers for running the selector on several GPUs of one node.

Rows are independent, so several GPUs never exchange data: each rank selects
its own batch (weak scaling) or its own contiguous range of a shared batch
(strong scaling).  The only collectives are for timing: a barrier around the
timed region and a max over ranks of the elapsed time.  They work with the
gloo backend on CPU tensors and with nccl on CUDA tensors.
"""

from __future__ import annotations


def row_range(rows: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced [start, end) of `rows` for `rank` of `world`."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own synthetic batch (distinct per rank)."""
    return int(seed) * 1_000_003 + int(rank)


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` across the default process group (identity if none)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()
