"""The N-rank host logic of bench.py on CPU: two gloo ranks, each with its own
time, agree on the slowest rank's time and report the whole-job rate; under
torchrun the reference arm runs on rank 0 only."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank  # rank 1 is slower
        ms_max, value = bench.job_throughput(ms_local, 2.0e12, 4, world)
        out[rank] = (ms_max, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank_and_the_job_rate():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    expect_ms = 15.0
    expect_value = world * 2.0e12 * 4 / (expect_ms / 1e3) / 1e12
    for rank in range(world):
        ms_max, value = out[rank]
        assert ms_max == pytest.approx(expect_ms)
        assert value == pytest.approx(expect_value)


def test_reference_arm_does_no_work_off_rank_zero():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        warmup, steps, cpu_rows = 1, 1, 64

    assert bench.run_reference(Args, rank=1) is None
