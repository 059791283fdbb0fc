"""The benchmark's multi-rank aggregation on CPU (gloo, two ranks): each rank
runs its own replica of the batch; the job's time is the slowest rank's and
its throughput counts every rank's units."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = [0.5, 2.0][rank]                       # rank 1 is the slow one
    out[rank] = (bench.max_over_ranks(t, world), bench.job_throughput(100.0, t, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_uses_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        mx, thr = res[rank]
        assert mx == 2.0
        assert thr == pytest.approx(100.0 * 2 / 2.0)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_throughput(10.0, 2.0, 1) == 5.0
