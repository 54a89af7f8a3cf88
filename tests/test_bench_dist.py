"""bench.py's multi-rank aggregation on CPU (gloo, world size 2): the
whole-job value is all ranks' steps over the slowest rank's time."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    value, slowest = bench.whole_job_value(0.5 + rank, 1000, world)
    bench.barrier(world)
    dist.destroy_process_group()
    q.put((rank, value, slowest))


def test_whole_job_value_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, value, slowest in res:
        assert slowest == pytest.approx(1.5)
        assert value == pytest.approx(2 * 1000 / 1.5)


def test_single_rank_identity():
    import bench
    assert bench.whole_job_value(2.0, 100, 1) == (50.0, 2.0)
