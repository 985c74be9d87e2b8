"""Multi-rank paths: one process per GPU.

Every (batch, head) of the attention is independent, so head-sharded inputs
need no data exchange: each rank runs its own problem (weak scaling) or its
own block of heads (`head_shard`, `head_sharded_sageattn`). Inputs sharded by
sequence, as Ulysses context parallelism holds them ("gfx1201 (RDNA4)
SageAttention attention backend: aiter package or Hub kernel?", sections
注意事项 and 解决步骤: the backend runs under Ulysses, inference only), take one
all-to-all from sequence shards to head blocks before the call and one back
after it (`ulysses_sageattn`). The exchanges go through torch.distributed
(NCCL on GPUs, gloo for the CPU tests of this logic); the attention itself is
the library's. Besides those, the only collectives are host-side
bookkeeping: a barrier around timed regions and the maximum of the ranks'
times.
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
    """The contiguous block [start, end) of n_heads that `rank` of `world`
    takes (of every batch): blocks differ in size by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must lie in [0, world)")
    base, extra = divmod(n_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def _nhd(t: torch.Tensor, tensor_layout: str) -> torch.Tensor:
    """t as a [B, S, H, D] view (HND tensors are transposed views)."""
    if tensor_layout == "NHD":
        return t
    if tensor_layout == "HND":
        return t.transpose(1, 2)
    raise ValueError(f"unknown tensor_layout {tensor_layout!r}")


def head_block(t: torch.Tensor, rank: int, world: int, tensor_layout: str = "NHD") -> torch.Tensor:
    """The view of t's heads that `rank` of `world` takes (no copy)."""
    x = _nhd(t, tensor_layout)
    s, e = head_shard(x.shape[2], rank, world)
    x = x[:, :, s:e]
    return x if tensor_layout == "NHD" else x.transpose(1, 2)


def head_sharded_sageattn(q, k, v, rank: int, world: int, tensor_layout: str = "NHD", is_causal: bool = False,
                          sm_scale=None, return_lse: bool = False, smooth_k: bool = True):
    """sageattn on this rank's block of heads of full q, k, v (each head is
    independent: no exchange). Returns the output of those heads in
    tensor_layout, and their log-sum-exp [B, heads, S] when return_lse."""
    from .api import sageattn, sageattn_ex

    qb, kb, vb = (head_block(t, rank, world, tensor_layout) for t in (q, k, v))
    if is_causal or return_lse:
        return sageattn_ex(qb, kb, vb, tensor_layout=tensor_layout, is_causal=is_causal, sm_scale=sm_scale,
                           return_lse=return_lse, smooth_k=smooth_k)
    return sageattn(qb, kb, vb, tensor_layout=tensor_layout, sm_scale=sm_scale, smooth_k=smooth_k)


def _group_info(group):
    import torch.distributed as dist

    if not dist.is_initialized():
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def _seq_lens(local_len: int, world: int, seq_lens):
    if seq_lens is None:
        return [local_len] * world
    seq_lens = [int(n) for n in seq_lens]
    if len(seq_lens) != world:
        raise ValueError("seq_lens needs one length per rank")
    return seq_lens


def ulysses_seq_to_heads(tensors, group=None, seq_lens=None) -> list:
    """All-to-all from sequence shards to head blocks. tensors: [B, S_r, H, D]
    tensors of this rank's sequence shard (S_r = seq_lens[rank]; by default
    every rank holds the same length). Returns, for each, [B, S, H_r, D] with
    S = sum(seq_lens): every rank's tokens, in rank order, of this rank's block
    of heads (head_shard). One exchange carries all the tensors."""
    import torch.distributed as dist

    world, rank = _group_info(group)
    if world == 1:
        return list(tensors)
    B, S_loc, H, D = tensors[0].shape
    lens = _seq_lens(S_loc, world, seq_lens)
    if lens[rank] != S_loc:
        raise ValueError("the local sequence shard does not match seq_lens")
    blocks = [head_shard(H, p, world) for p in range(world)]
    # send: per destination p, its head block of every tensor
    send = torch.cat([t[:, :, s:e].reshape(-1) for s, e in blocks for t in tensors])
    send_sizes = [len(tensors) * B * S_loc * (e - s) * D for s, e in blocks]
    hs, he = blocks[rank]
    recv_sizes = [len(tensors) * B * n * (he - hs) * D for n in lens]
    recv = torch.empty(sum(recv_sizes), dtype=send.dtype, device=send.device)
    dist.all_to_all_single(recv, send, recv_sizes, send_sizes, group=group)
    out = []
    parts = recv.split(recv_sizes)
    for i in range(len(tensors)):
        pieces = [part.view(len(tensors), B, n, he - hs, D)[i] for part, n in zip(parts, lens)]
        out.append(torch.cat(pieces, dim=1))
    return out


def ulysses_heads_to_seq(y: torch.Tensor, n_heads: int, group=None, seq_lens=None) -> torch.Tensor:
    """All-to-all back from head blocks to sequence shards: y [B, S, H_r, D]
    (this rank's heads, every token) -> [B, S_r, n_heads, D] (this rank's
    tokens, every head)."""
    import torch.distributed as dist

    world, rank = _group_info(group)
    if world == 1:
        return y
    B, S, Hr, D = y.shape
    lens = _seq_lens(S // world, world, seq_lens)
    if sum(lens) != S:
        raise ValueError("seq_lens must add up to the full sequence")
    starts = [sum(lens[:p]) for p in range(world)]
    blocks = [head_shard(n_heads, p, world) for p in range(world)]
    send = torch.cat([y[:, a:a + n].reshape(-1) for a, n in zip(starts, lens)])
    send_sizes = [B * n * Hr * D for n in lens]
    recv_sizes = [B * lens[rank] * (e - s) * D for s, e in blocks]
    recv = torch.empty(sum(recv_sizes), dtype=send.dtype, device=send.device)
    dist.all_to_all_single(recv, send, recv_sizes, send_sizes, group=group)
    out = torch.empty((B, lens[rank], n_heads, D), dtype=y.dtype, device=y.device)
    for part, (s, e) in zip(recv.split(recv_sizes), blocks):
        out[:, :, s:e] = part.view(B, lens[rank], e - s, D)
    return out


def ulysses_lse_to_seq(lse: torch.Tensor, n_heads: int, group=None, seq_lens=None) -> torch.Tensor:
    """The log-sum-exp of this rank's heads over every token, [B, H_r, S],
    back to this rank's tokens of every head, [B, n_heads, S_r]."""
    import torch.distributed as dist

    world, rank = _group_info(group)
    if world == 1:
        return lse
    B, Hr, S = lse.shape
    lens = _seq_lens(S // world, world, seq_lens)
    starts = [sum(lens[:p]) for p in range(world)]
    blocks = [head_shard(n_heads, p, world) for p in range(world)]
    send = torch.cat([lse[:, :, a:a + n].reshape(-1) for a, n in zip(starts, lens)])
    send_sizes = [B * Hr * n for n in lens]
    recv_sizes = [B * (e - s) * lens[rank] for s, e in blocks]
    recv = torch.empty(sum(recv_sizes), dtype=send.dtype, device=send.device)
    dist.all_to_all_single(recv, send, recv_sizes, send_sizes, group=group)
    out = torch.empty((B, n_heads, lens[rank]), dtype=lse.dtype, device=lse.device)
    for part, (s, e) in zip(recv.split(recv_sizes), blocks):
        out[:, s:e] = part.view(B, e - s, lens[rank])
    return out


def ulysses_sageattn(q, k, v, group=None, tensor_layout: str = "NHD", is_causal: bool = False, sm_scale=None,
                     return_lse: bool = False, smooth_k: bool = True, seq_lens=None):
    """sageattn over a sequence sharded across the ranks of `group` (Ulysses):
    q, k, v hold this rank's tokens of every head ([B, S_r, H, D] in NHD,
    [B, H, S_r, D] in HND). One all-to-all gathers, for this rank's block of
    heads, every rank's tokens; the library's sageattn runs on them (the
    causal mask and the log-sum-exp see the whole sequence); one all-to-all
    returns each rank its tokens of every head. Returns this rank's output
    (and log-sum-exp [B, H, S_r] when return_lse) in tensor_layout. With one
    rank, or no process group, it is sageattn itself."""
    from .api import sageattn, sageattn_ex

    world, _ = _group_info(group)
    if world == 1:
        if is_causal or return_lse:
            return sageattn_ex(q, k, v, tensor_layout=tensor_layout, is_causal=is_causal, sm_scale=sm_scale,
                               return_lse=return_lse, smooth_k=smooth_k)
        return sageattn(q, k, v, tensor_layout=tensor_layout, sm_scale=sm_scale, smooth_k=smooth_k)
    qn, kn, vn = (_nhd(t, tensor_layout) for t in (q, k, v))
    H = qn.shape[2]
    qh, kh, vh = ulysses_seq_to_heads([qn, kn, vn], group, seq_lens)
    if is_causal or return_lse:
        res = sageattn_ex(qh, kh, vh, tensor_layout="NHD", is_causal=is_causal, sm_scale=sm_scale,
                          return_lse=return_lse, smooth_k=smooth_k)
    else:
        res = sageattn(qh, kh, vh, tensor_layout="NHD", sm_scale=sm_scale, smooth_k=smooth_k)
    out_h, lse_h = (res if return_lse else (res, None))
    out = ulysses_heads_to_seq(out_h, H, group, seq_lens)
    if tensor_layout == "HND":
        out = out.transpose(1, 2).contiguous()
    if return_lse:
        return out, ulysses_lse_to_seq(lse_h, H, group, seq_lens)
    return out


def teardown(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
