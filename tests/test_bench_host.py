"""Host-side logic of bench.py's multi-process path, run as two gloo ranks on
the CPU: the timed region is the slowest rank's, and the whole-job value
counts every replica's work."""
import os
import socket

import pytest
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


REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "cpu_baseline", "e2e", "impl"}


@pytest.mark.parametrize("args", [["--workload", "1"], ["--op", "quantize", "--qworkload", "1"]],
                         ids=["gemm", "quantize"])
def test_reference_arm_prints_one_contract_line(args):
    """`bench.py --impl reference` times the oracle on the host and prints one
    JSON line with the contract's keys, the metric of the GPU arm and an e2e
    entry with no host-device copies."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-seconds", "1", *args], cwd=root,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert REQUIRED <= set(d), REQUIRED - set(d)
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["metric"] == (bench.QMETRIC if "quantize" in args else bench.METRIC)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_traffic_key_ignores_comments_but_not_code(tmp_path, monkeypatch):
    """The ncu traffic reported in the roofline is keyed by a hash of the
    kernel source without comments and whitespace: editing a comment keeps the
    captured counters valid, changing code makes the lookup miss (null)."""
    src = os.path.join(bench.ROOT, "block_scaled_precision_04_gb300", "csrc", "bsgemm.cu")
    text = open(src).read()
    csrc = tmp_path / "block_scaled_precision_04_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "bsgemm.cu").write_text(text)
    h0 = bench.kernel_source_hash()
    (csrc / "bsgemm.cu").write_text("// a new comment\n" + text.replace("\n", "\n  ", 3))
    assert bench.kernel_source_hash() == h0
    (csrc / "bsgemm.cu").write_text(text.replace("kRnd = 4", "kRnd = 2", 1))
    assert bench.kernel_source_hash() != h0
    assert all(len(k[0]) == 16 for k in bench.TRAFFIC)


def test_host_cost_is_a_burst_of_launches():
    """The host cost per launch is the wall time of n launches enqueued back
    to back, divided by n, with the device synchronised on both sides."""
    import types
    calls, syncs = [], []
    fake_torch = types.SimpleNamespace(cuda=types.SimpleNamespace(synchronize=lambda d: syncs.append(d)))
    us = bench.host_cost_us(lambda: calls.append(1), fake_torch, "dev", n=50)
    assert len(calls) == 50 and syncs == ["dev", "dev"]
    assert isinstance(us, float) and 0.0 <= us < 1e4


def test_local_piece_single_gpu_is_the_workload():
    import numpy as np
    import synth
    g, inp, piece = bench.local_piece(1, 1, 0, "batches")
    assert piece is None and g == synth.WORKLOADS[1][1]
    assert np.array_equal(inp.A, synth.workload(1).A)


def test_local_piece_batches_weak_scaling():
    """--shard batches: the global problem repeats the workload's L batches
    once per rank; rank r owns batches [r L, (r+1) L), drawn from a seed of
    its own (rank 0's are the workload itself)."""
    import numpy as np
    import synth
    p = synth.WORKLOADS[1][1]
    pieces = [bench.local_piece(1, 3, r, "batches") for r in range(3)]
    for r, (g, inp, s) in enumerate(pieces):
        assert g.L == 3 * p.L and (g.M, g.N, g.K) == (p.M, p.N, p.K)
        assert (s.l0, s.l1, s.m0, s.m1) == (r * p.L, (r + 1) * p.L, 0, p.M)
        assert inp.problem == p
    assert np.array_equal(pieces[0][1].A, synth.workload(1).A)
    assert not np.array_equal(pieces[0][1].A, pieces[1][1].A)
    assert len({bench.batch_seed(1, r) for r in range(8)}) == 8


def test_local_piece_rows_strong_scaling():
    """--shard rows: the ranks split the workload's rows in whole 128-row
    scale atoms; each piece is the workload's own rows and scale atoms."""
    import numpy as np
    import synth
    full = synth.workload(1)
    got = []
    for r in range(2):
        g, inp, s = bench.local_piece(1, 2, r, "rows")
        assert g == full.problem and inp.problem.M == s.rows
        assert np.array_equal(inp.A, full.A[:, s.m0:s.m1])
        assert np.array_equal(inp.B, full.B) and np.array_equal(inp.SFB, full.SFB)
        assert np.array_equal(inp.SFA, full.SFA[:, s.m0 // 128:-(-s.m1 // 128)])
        got.append((s.m0, s.m1))
    assert got == [(0, 128), (128, 256)]


def test_gpus_flag_must_match_world_size(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    assert bench.main(["--gpus", "4", "--impl", "reference"]) == 2
    assert "WORLD_SIZE 2" in capsys.readouterr().err
