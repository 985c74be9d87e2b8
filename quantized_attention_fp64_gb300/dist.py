"""Multi-rank host logic: one process per GPU, replicas of the workload.

Every (batch, head) of the attention is independent, so ranks need no data
exchange: each rank runs its own problem (weak scaling) or its own block of
heads (`head_shard`). The only collectives are host-side bookkeeping: a
barrier around timed regions and the maximum of the ranks' times. NCCL on
GPUs, gloo for the CPU tests of this logic.
"""

from __future__ import annotations

import os

import torch


def setup(backend: str | None = None):
    """(rank, world, local_rank) from the launcher's environment (RANK,
    WORLD_SIZE, LOCAL_RANK, MASTER_ADDR/PORT); joins the process group when
    world > 1. backend None: NCCL with the local GPU as the rank's device."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if backend is None or backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend is None:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over the ranks (a time: the job ends with its slowest rank)."""
    if world == 1:
        return x
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def head_shard(n_heads: int, rank: int, world: int) -> tuple[int, int]:
    """The contiguous block [start, end) of n_heads (batch-major (b, h) pairs)
    that `rank` of `world` takes: blocks differ in size by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must lie in [0, world)")
    base, extra = divmod(n_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def teardown(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
