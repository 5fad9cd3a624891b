"""Multi-rank bench logic on CPU: two gloo ranks (replicas) agree on the max
time and on the whole-job throughput; no data-path collective exists."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [0.25, 0.5][rank]                    # rank 1 is the slow replica
        m = bench.dist_max(local, world)
        v = bench.job_throughput(world, 177, 10, m)
        out[rank] = (m, v)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_max_and_sum_replicas():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    m, v = out[0]
    assert m == 0.5
    assert v == pytest.approx(2 * 177 * 10 / 0.5)


def test_single_rank_passthrough():
    import bench
    assert bench.dist_max(1.5, 1) == 1.5
    assert bench.job_throughput(1, 177, 40, 2.0) == 177 * 40 / 2.0
