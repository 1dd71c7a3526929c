"""The multi-GPU path is replicas only: every rank runs its own copy of the
workload and the bench takes the slowest rank's time.  This checks that
reduction over two gloo ranks on the CPU."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.barrier_max(1.5 + rank, world)
    q.put((rank, t))
    dist.destroy_process_group()


def test_slowest_rank_time_is_reported():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


@pytest.mark.parametrize("world", [1])
def test_single_rank_is_identity(world):
    import bench
    assert bench.barrier_max(3.25, world) == 3.25
