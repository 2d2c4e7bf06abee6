"""Host-side logic of bench.py's multi-process path, run as two gloo ranks on
the CPU: the timed region is the slowest rank's, and the whole-job value
counts every replica's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        out[rank] = slowest
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5) == 3.5


def test_whole_job_value_counts_every_replica():
    flops = 2.0 * 4096 ** 3
    one = bench.whole_job_tflops(flops, 10, 1, 1.0)
    assert one == pytest.approx(flops * 10 / 1e-3 / 1e12)
    assert bench.whole_job_tflops(flops, 10, 4, 1.0) == pytest.approx(4 * one)


def test_workload_numbers_match_the_page_sizes():
    import synth
    _, p = synth.WORKLOADS[2]
    n = bench.workload_numbers(p)
    assert n["flops"] == 2.0 * 4096 ** 3
    # A + B (1 byte per code) + padded scale atoms + bf16 C
    sf = 32 * 32 * 512
    assert n["bytes"] == 2 * 4096 * 4096 + 2 * sf + 2 * 4096 * 4096
    assert n["kind"] == "fp8"
