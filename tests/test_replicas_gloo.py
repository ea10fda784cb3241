"""The N-replica path of bench.py on the CPU: two gloo ranks with different
step times; the job's step time is the slower rank's and the throughput
counts both ranks' tokens (weak scaling, no data-path collective)."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = 2.0 if rank == 0 else 3.0          # rank 1 is the slow replica
        ms, value = bench.aggregate(step_ms, 31, world)
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    port = 29500 + os.getpid() % 1000
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        ms, value = res[rank]
        assert ms == pytest.approx(3.0)
        assert value == pytest.approx(2 * 31 / 0.003)


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(2.0, 31, 1) == (2.0, pytest.approx(31 / 0.002))
