"""The N>1 path of bench.py (independent replicas, one per GPU): every rank
ends up with the slowest rank's timings and the whole-job rate counts the work
of all replicas.  Run as two gloo processes on the CPU."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
    got = bench.max_over_ranks(local, dist)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_with_gloo(world):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    expect = [float(world), 5.0, 0.25 * world]
    for r in range(world):
        assert list(out[r]) == expect


def test_max_over_ranks_without_process_group_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.0]) == [1.5, 2.0]


def test_job_rate_counts_all_replicas():
    import bench
    assert bench.job_rate(10.0, 4, 2.0) == 20.0
