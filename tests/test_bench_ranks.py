"""Host logic of bench.py's multi-GPU launch (CPU, gloo, world size 2): each
rank times its own replica; the job time is the maximum over ranks and the
job value counts the work of all ranks."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank)           # rank 1 is the slow one
    out[rank] = (ms, bench.job_value(2e12, world, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, value = out[r]
        assert ms == 15.0
        assert value == pytest.approx(2e12 * 2 / 15e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(1e12, 1, 1.0) == pytest.approx(1000.0)
