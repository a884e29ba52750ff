"""The N > 1 path of the benchmark is replicas only: every rank runs its own
copy of the workload, the job's time is the slowest rank's (max over ranks)
and the job's throughput is the units of all ranks over that time.  These
two pieces are exercised here with two gloo ranks on the CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = [1.5, 4.0][rank]          # per-rank step times
    job_ms = bench.max_over_ranks(my_ms, dist)
    rate = bench.job_throughput(1e12, world, job_ms)
    out[rank] = (job_ms, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        job_ms, rate = out[r]
        assert job_ms == 4.0                      # both ranks see the slowest time
        assert rate == pytest.approx(2 * 1.0 / 4e-3)  # 2 ranks x 1 TFLOP per 4 ms


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(2.5, None) == 2.5
    assert bench.job_throughput(2e12, 1, 1.0) == pytest.approx(2000.0)
