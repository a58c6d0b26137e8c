"""The multi-rank timing path of bench.py on CPU: two gloo ranks, each with
its own time; both must see the maximum, and the whole-job value must count
the work of both ranks over that time."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = bench.max_over_ranks(times[rank], dist, "cpu")
    value = bench.whole_job_tflops(10 ** 12, world, ms)
    dist.barrier()
    results[rank] = (ms, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    times = [12.5, 17.25]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        ms, value = results[r]
        assert ms == 17.25
        assert value == pytest.approx(2 * 10 ** 12 / 17.25e-3 / 1e12)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(4 * 10 ** 12, 1, 1000.0) == pytest.approx(4.0)
