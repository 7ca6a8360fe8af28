"""The multi-rank path of bench.py on CPU: two gloo ranks take the maximum of
their step times (the slowest replica sets the job's step time) and the job
throughput counts every rank's work (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1.0 + rank, 10.0 - rank]          # rank 1 slower on the first value
    got = bench.max_over_ranks(mine, dist, "cpu")
    results[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        assert results[0] == [2.0, 10.0] and results[1] == [2.0, 10.0]


def test_job_throughput_counts_every_replica():
    import bench
    one = bench.job_throughput(bench.STEP_FLOPS, 1, 2.0)
    assert bench.job_throughput(bench.STEP_FLOPS, 4, 2.0) == pytest.approx(4 * one)
    assert one == pytest.approx(bench.STEP_FLOPS / 2e-3 / 1e12)
