"""The N>1 path of the benchmark on the CPU: two gloo ranks run their own
replica and combine only their timings. The job's time is the slowest rank's,
and its throughput counts the units of every rank."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_deltanet_linear_02_gb300.replicas import job_rate, slowest_ms


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]                 # rank 1 is the slow one
        job_ms = slowest_ms(local_ms)
        out[rank] = (job_ms, job_rate(256 * 32, world, job_ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:       # no fork from this multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]                          # every rank agrees
    job_ms, rate = res[0]
    assert job_ms == 20.0
    assert rate == pytest.approx(2 * 256 * 32 / 0.020)


def test_single_process_passes_through():
    assert slowest_ms(7.0) == 7.0
    assert job_rate(100, 1, 50.0) == pytest.approx(2000.0)
    with pytest.raises(ValueError):
        job_rate(1, 1, 0.0)
