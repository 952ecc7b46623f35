"""Host-side multi-rank logic (gloo, world size 2, CPU): the benchmark's replicas
aggregate to N x tokens over the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 100.0 * (rank + 1)  # rank 1 is the slow one
    value, total_ms = bench.aggregate_throughput(local_ms, 1000.0, dist, "cpu")
    out[rank] = (value, total_ms)
    dist.destroy_process_group()


def test_replicas_aggregate_over_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        value, total_ms = res[rank]
        assert total_ms == pytest.approx(200.0)
        assert value == pytest.approx(world * 1000.0 / 0.2)


def test_single_process_aggregate():
    import bench

    value, total_ms = bench.aggregate_throughput(50.0, 500.0)
    assert total_ms == 50.0 and value == pytest.approx(10000.0)
