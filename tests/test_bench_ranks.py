"""Replica timing logic of bench.py with two ranks on CPU (gloo): every rank sees the
slowest rank's time, and the job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slow = bench.max_over_ranks(1.0 + 2.0 * rank, world)          # rank 1 is slower: 3.0 ms
    q.put((rank, slow, bench.job_throughput(16, world, slow)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, value in got:
        assert slow == pytest.approx(3.0)
        assert value == pytest.approx(2 * 16 / 3.0e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_throughput(16, 1, 0.5) == pytest.approx(32000.0)
