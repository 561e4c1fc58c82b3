"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank
times its own batch, the job time is the slowest rank's, and the whole-job
throughput counts every rank's work once."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


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
