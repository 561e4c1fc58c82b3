"""Multi-rank host logic on CPU (gloo, world size 2).

bench.py: each rank times its work, the job time is the slowest rank's, and
the whole-job throughput counts every rank's work once.  The head partition
(bit_attention_gb300.shard): the ranks' shares cover every (batch, head)
exactly once, and gathering O puts every head's rows back in order."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_attention_gb300.shard import gather_heads, head_view, shard_heads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = 10.0 + 5.0 * rank          # rank 1 is slower
    t = bench.max_over_ranks(my_ms, world)
    bench.barrier(world)
    q.put((rank, t, bench.job_throughput(1e12, world, t)))
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in out:
        assert t == 15.0                      # both ranks agree on the slowest time
        assert v == pytest.approx(2 * 1e12 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(2e12, 1, 2.0) == pytest.approx(1000.0)


# ---------------------------------------------------------------- head partition

@pytest.mark.parametrize("B,H,world", [(4, 32, 2), (4, 32, 8), (2, 48, 3), (1, 3, 8), (3, 5, 4),
                                       (1, 1, 1), (0, 4, 2)])
def test_shards_cover_every_head_exactly_once(B, H, world):
    seen = []
    for r in range(world):
        first, count = shard_heads(B, H, r, world)
        assert count >= 0
        seen.extend(range(first, first + count))
    assert seen == list(range(B * H))  # every head once, in rank order
    counts = [shard_heads(B, H, r, world)[1] for r in range(world)]
    assert max(counts) - min(counts) <= 1


def test_head_view_is_the_contiguous_slab_of_those_heads():
    x = torch.arange(2 * 3 * 4 * 8, dtype=torch.float32).reshape(2, 3, 4, 8)
    v = head_view(x, 2, 3)  # heads (0,2), (1,0), (1,1)
    assert v.shape == (1, 3, 4, 8) and v.data_ptr() == x[0, 2].data_ptr()
    assert torch.equal(v[0], torch.stack([x[0, 2], x[1, 0], x[1, 1]]))


def _gather_worker(rank, world, port, B, H, N, D, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    first, count = shard_heads(B, H, rank, world)
    # byte-tagged O share: element (head j, token n, channel d) holds
    # 1000 * (global head) + 10 * n + d, so any misplaced row shows
    heads = torch.arange(first, first + count, dtype=torch.float32)[:, None, None]
    n = torch.arange(N, dtype=torch.float32)[None, :, None]
    d = torch.arange(D, dtype=torch.float32)[None, None, :]
    local = (1000 * heads + 10 * n + d).unsqueeze(0)
    full = gather_heads(local, B, H)
    q.put((rank, full.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("B,H", [(2, 3), (1, 4)])
def test_two_rank_gather_puts_heads_back_in_order(B, H):
    world, N, D = 2, 5, 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, B, H, N, D, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import numpy as np
    j = np.arange(B * H, dtype=np.float32).reshape(B, H, 1, 1)
    want = 1000 * j + 10 * np.arange(N, dtype=np.float32)[None, None, :, None] + \
        np.arange(D, dtype=np.float32)[None, None, None, :]
    for _, full in out:
        assert full.shape == (B, H, N, D)
        assert np.array_equal(full, want)
