"""The multi-rank host logic on CPU: two gloo ranks (one process each) join
through the launcher's environment, meet at the barrier, agree on the largest
time and split heads into blocks with no data exchange. The attention itself
needs no collective: every (batch, head) is independent."""

import os
import socket

import pytest
import torch.multiprocessing as mp

from quantized_attention_fp64_gb300 import dist


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    r, w, local = dist.setup("gloo")
    assert (r, w, local) == (rank, world, rank)
    dist.barrier(w)
    t = dist.max_over_ranks(times[rank], w, device="cpu")
    shard = dist.head_shard(28, r, w)
    dist.barrier(w)
    dist.teardown(w)
    queue.put((rank, t, shard))


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_agree_on_the_slowest_time_and_split_heads(world):
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    times = [1.25 + 0.5 * r for r in range(world)]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, queue)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [t for _, t, _ in results] == [max(times)] * world
    shards = [s for _, _, s in results]
    assert shards[0][0] == 0 and shards[-1][1] == 28
    assert all(a[1] == b[0] for a, b in zip(shards, shards[1:]))
    assert max(e - s for s, e in shards) - min(e - s for s, e in shards) <= 1


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert dist.setup("gloo") == (0, 1, 0)
    assert dist.max_over_ranks(3.5, 1) == 3.5
    dist.barrier(1)
    dist.teardown(1)


@pytest.mark.parametrize("n,world", [(28, 2), (28, 3), (5, 8), (0, 4), (1, 1)])
def test_head_shard_covers_every_head_once(n, world):
    blocks = [dist.head_shard(n, r, world) for r in range(world)]
    covered = [h for s, e in blocks for h in range(s, e)]
    assert covered == list(range(n))
    with pytest.raises(ValueError):
        dist.head_shard(n, world, world)


# --------------------------------------------------------------------------
# Ulysses (sequence-sharded) exchanges and the head-sharded split, on gloo
# ranks. The attention between the exchanges is the oracle's exact fp64
# attention here (the library's kernels need a GPU); its result for the
# gathered head blocks, sent back to the sequence shards, must equal the
# oracle's attention of the whole tensors bit for bit, since every head is
# computed from the same values in the same order.

def _global_qkv(B, S, H, D, seed=7):
    import numpy as np

    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B, S, H, D)) for _ in range(3)]


def _ulysses_rank_main(rank, world, port, lens, H, causal, queue):
    import numpy as np
    import torch

    from oracle.tensors import exact_head

    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    r, w, _ = dist.setup("gloo")
    B, D, S = 2, 8, sum(lens)
    q, k, v = _global_qkv(B, S, H, D)
    a = sum(lens[:r])
    shard = [torch.from_numpy(x[:, a:a + lens[r]].copy()) for x in (q, k, v)]
    gathered = dist.ulysses_seq_to_heads(shard, None, lens)
    hs, he = dist.head_shard(H, r, w)
    ok_gather = all(torch.equal(g, torch.from_numpy(x[:, :, hs:he].copy())) for g, x in zip(gathered, (q, k, v)))
    back = dist.ulysses_heads_to_seq(gathered[0], H, None, lens)
    ok_round = torch.equal(back, shard[0])
    # attention of this rank's heads over every token (oracle), then back to
    # this rank's tokens of every head
    qh, kh, vh = (g.numpy() for g in gathered)
    sm = 1.0 / np.sqrt(D)
    y = np.zeros((B, S, he - hs, D))
    lse_h = np.zeros((B, he - hs, S))
    for b in range(B):
        for hh in range(he - hs):
            y[b, :, hh], lse_h[b, hh] = exact_head(qh, kh, vh, "NHD", sm, b, hh, causal=causal, return_lse=True)
    out = dist.ulysses_heads_to_seq(torch.from_numpy(y), H, None, lens).numpy()
    lse = dist.ulysses_lse_to_seq(torch.from_numpy(lse_h), H, None, lens).numpy()
    ref = np.zeros((B, lens[r], H, D))
    ref_lse = np.zeros((B, H, lens[r]))
    for b in range(B):
        for h in range(H):
            o, l_ = exact_head(q, k, v, "NHD", sm, b, h, causal=causal, return_lse=True)
            ref[b, :, h], ref_lse[b, h] = o[a:a + lens[r]], l_[a:a + lens[r]]
    dist.barrier(w)
    dist.teardown(w)
    queue.put((rank, ok_gather, ok_round, bool(np.array_equal(out, ref)), bool(np.array_equal(lse, ref_lse))))


@pytest.mark.parametrize("world,lens,H,causal", [(2, [6, 6], 5, False), (3, [4, 4, 4], 7, True),
                                                  (2, [5, 3], 4, True)])
def test_ulysses_exchanges_and_attention_match_the_whole_tensors(world, lens, H, causal):
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ulysses_rank_main, args=(r, world, port, lens, H, causal, queue))
             for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ok_gather, ok_round, ok_out, ok_lse in results:
        assert ok_gather, f"rank {rank}: gathered head block differs"
        assert ok_round, f"rank {rank}: round trip differs"
        assert ok_out, f"rank {rank}: attention output differs from the whole-tensor oracle"
        assert ok_lse, f"rank {rank}: log-sum-exp differs from the whole-tensor oracle"


@pytest.mark.parametrize("world,H", [(2, 5), (3, 7), (4, 3)])
def test_head_blocks_join_to_the_whole_tensor(world, H):
    import numpy as np
    import torch

    B, S, D = 2, 9, 8
    x = torch.from_numpy(_global_qkv(B, S, H, D)[0])
    blocks = [dist.head_block(x, r, world) for r in range(world)]
    assert torch.equal(torch.cat(blocks, dim=2), x)
    xh = x.transpose(1, 2).contiguous()   # HND
    blocks_h = [dist.head_block(xh, r, world, "HND") for r in range(world)]
    assert torch.equal(torch.cat(blocks_h, dim=1), xh)
    assert all(b.data_ptr() == x[:, :, dist.head_shard(H, r, world)[0]:].data_ptr() for r, b in enumerate(blocks))
    assert np.all([b.shape[2] for b in blocks] == np.diff([dist.head_shard(H, r, world)[0] for r in range(world)]
                                                           + [H]))
