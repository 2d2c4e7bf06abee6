"""The sharded form on one GPU: every rank's piece (whole batches, or whole
128-row scale atoms of one batch) launched one after another through the C
ABI into views of one C, then Amax reduced over the pieces.  The pieces are
independent launches that never wait on one another.  The assembled C must
pass the oracle parity check and the reduced Amax must equal max |C|."""
import os
import socket

import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import synth
from block_scaled_precision_04_gb300 import shard as sh
from gpu_util import TORCH_C, abs_max_bits, assert_parity, c_to_logical, problem_of, to_device

pytestmark = pytest.mark.gpu

CASES = [
    (synth.Problem(512, 640, 256, 4, "e4m3", "e5m2", 32, "bf16", "n"), 3),           # batches
    (synth.Problem(1000, 520, 384, 1, "e2m1", "e2m1", 16, "f32", "n"), 3),           # rows
    (synth.Problem(700, 384, 256, 2, "e4m3", "e4m3", 32, "bf16", "n"), 5),           # mixed
    (synth.Problem(1000, 512, 384, 1, "e2m1", "e2m1", 16, "e2m1", "n"), 4),          # rows, FP4 C
    (synth.Problem(304, 256, 128, 3, "e4m3", "e4m3", 32, "f16", "m", a_major="m",
                   b_major="n"), 3),                                                    # batches, MN-major
]


@pytest.mark.parametrize("p,world", CASES, ids=lambda x: x.describe().replace(" ", "_")
                         if isinstance(x, synth.Problem) else str(x))
def test_sharded_pieces_assemble_the_whole(p, world):
    inp = synth.uniform_codes(p, p.M + p.L * world, 120, 128)
    A, B, SFA, SFB = to_device(inp)
    C = torch.empty(synth.c_shape(p), dtype=TORCH_C[p.c_dtype], device="cuda:0")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda:0")
    for r in range(world):
        s = sh.shard_of(p.M, p.L, world, r)
        if s.empty:
            continue
        a, b, sfa, sfb, c = sh.local_views(s, A, B, SFA, SFB, C, M=p.M, a_major=p.a_major,
                                           c_major=p.c_major)
        op = bsg.GemmAmax(problem_of(sh.local_problem(p, s)))
        local = torch.zeros(1, dtype=torch.float32, device="cuda:0")
        op.run(a, b, sfa, sfb, c, local)
        torch.cuda.synchronize()
        assert op.device_status() == bsg.BSG_OK
        # the all-reduce's integer max, here over the pieces in turn
        amax.view(torch.int32).copy_(torch.maximum(amax.view(torch.int32), local.view(torch.int32)))
    c_full = c_to_logical(C, p)
    assert np.float32(amax.item()).view(np.uint32) == abs_max_bits(c_full)
    assert_parity(inp, c_full, float(amax.item()))


def _nccl_single_rank(rank, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        amax = torch.tensor([3.25], dtype=torch.float32, device="cuda:0")
        sh.allreduce_amax(amax)
        nan = torch.tensor([float("nan")], dtype=torch.float32, device="cuda:0")
        sh.allreduce_amax(nan)
        torch.cuda.synchronize()
        out["amax"] = float(amax.item())
        out["nan_bits"] = int(nan.view(torch.int32).item()) & 0xFFFFFFFF
    finally:
        dist.destroy_process_group()


def test_nccl_allreduce_amax_single_rank():
    """The multi-GPU exchange's own call path on NCCL: a one-rank group on
    this GPU reduces the fp32 Amax as an int32 max in place (the value and a
    NaN's bits come back unchanged).  Run in a spawned process so that the
    group leaves no state behind."""
    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_nccl_single_rank, args=(port, out), nprocs=1, join=True,
                       start_method="spawn")
    assert out["amax"] == 3.25
    assert out["nan_bits"] == 0x7FC00000
