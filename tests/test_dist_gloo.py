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
