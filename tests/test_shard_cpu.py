"""The sharded form of the GEMM + Amax over gloo ranks on the CPU: every rank
computes its piece (here with the oracle, standing in for the rank's GPU),
the ranks all-reduce Amax, and the assembled pieces equal the unsharded
result.  Pieces follow the partition the library's shard module defines:
whole batches, or whole 128-row scale atoms of one batch."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
from block_scaled_precision_04_gb300 import shard as sh


# ------------------------------------------------------------ partition

@pytest.mark.parametrize("M,L,world", [(1, 1, 1), (300, 4, 2), (300, 8, 3), (1000, 1, 4),
                                       (1000, 2, 3), (100, 1, 2), (4096, 3, 8), (129, 5, 5)])
def test_partition_covers_every_element_once(M, L, world):
    owner = np.full((L, M), -1)
    for r in range(world):
        s = sh.shard_of(M, L, world, r)
        if s.empty:
            continue
        assert s.m0 % sh.ATOM_ROWS == 0 and (s.m1 == M or s.m1 % sh.ATOM_ROWS == 0)
        assert np.all(owner[s.l0:s.l1, s.m0:s.m1] == -1)
        owner[s.l0:s.l1, s.m0:s.m1] = r
    assert np.all(owner >= 0)


def test_partition_balance():
    # whole batches: sizes differ by at most one batch
    sizes = [sh.shard_of(64, 8, 3, r).batches for r in range(3)]
    assert sorted(sizes) == [2, 3, 3]
    # rows: in whole atoms, differing by at most one atom
    rows = [sh.shard_of(4096, 1, 3, r).rows for r in range(3)]
    assert sum(rows) == 4096 and max(rows) - min(rows) <= sh.ATOM_ROWS
    # more ranks than atoms leaves some ranks empty
    assert sorted(sh.shard_of(100, 1, 2, r).empty for r in range(2)) == [False, True]


def test_row_split_needs_contiguous_rows():
    p = synth.Problem(300, 64, 64, 1, "e4m3", "e4m3", 32, "f32", "m")
    inp = synth.uniform_codes(p, 1)
    s = sh.shard_of(p.M, p.L, 2, 0)
    C = np.zeros(synth.c_shape(p), dtype=np.float32)
    with pytest.raises(ValueError):
        sh.local_views(s, inp.A, inp.B, inp.SFA, inp.SFB, C, M=p.M, c_major="m")


@pytest.mark.parametrize("M,L,world,a,c", [(300, 4, 3, "e4m3", "f32"), (1000, 1, 4, "e4m3", "bf16"),
                                           (520, 2, 5, "e2m1", "f16"), (100, 1, 2, "e2m1", "bf16")])
def test_views_span_the_local_problem(M, L, world, a, c):
    """Each rank's views hold exactly the bytes its local problem spans (the
    binding's size check on a run), are C-contiguous (a plain pointer and the
    library's strides describe them) and start where the rank's rows do."""
    import block_scaled_precision_04_gb300 as bsg
    sfv = 16 if a == "e2m1" else 32
    p = synth.Problem(M, 160, 256, L, a, a, sfv, c, "n")
    inp = synth.uniform_codes(p, M + world)
    C = np.zeros(synth.c_shape(p), dtype=np.float32 if c == "f32" else np.uint16)
    full = bsg.make_problem(p.M, p.N, p.K, p.L, a, a, sfv, c, "n")
    for r in range(world):
        s = sh.shard_of(M, L, world, r)
        if s.empty:
            continue
        views = sh.local_views(s, inp.A, inp.B, inp.SFA, inp.SFB, C, M=M)
        need = bsg.problem_bytes(sh.local_problem(full, s))
        for key, v in zip(("A", "B", "SFA", "SFB", "C"), views):
            assert v.flags["C_CONTIGUOUS"], key
            assert v.nbytes == need[key], (key, r)
        a_view, c_view = views[0], views[4]
        row0 = (s.l0 * M + s.m0)
        assert a_view.ctypes.data - inp.A.ctypes.data == row0 * inp.A.shape[-1]
        assert c_view.ctypes.data - C.ctypes.data == row0 * C.shape[-1] * C.itemsize


# ------------------------------------------------------------- gloo ranks

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = {
    "batches": synth.Problem(200, 96, 64, 4, "e4m3", "e5m2", 32, "bf16", "n"),
    "rows": synth.Problem(300, 80, 96, 1, "e2m1", "e2m1", 16, "f32", "n"),
    "mixed": synth.Problem(260, 64, 64, 2, "e4m3", "e4m3", 32, "f32", "n"),
    "empty rank": synth.Problem(100, 48, 64, 1, "e4m3", "e4m3", 32, "f16", "n"),
}


def _rank(rank, world, port, name, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = CASES[name]
        inp = synth.uniform_codes(p, 11, 118, 132)   # every rank draws the same inputs
        s = sh.shard_of(p.M, p.L, world, rank)
        amax = torch.zeros(1, dtype=torch.float32)
        piece = None
        if not s.empty:
            C = np.zeros(synth.c_shape(p), dtype=np.float32)
            A, B, SFA, SFB, _ = sh.local_views(s, inp.A, inp.B, inp.SFA, inp.SFB, C, M=p.M)
            lp = sh.local_problem(p, s)
            ref = oracle.reference(lp.M, lp.N, lp.K, lp.L, lp.a_dtype, lp.b_dtype, lp.sfv, A, B,
                                   SFA, SFB, lp.c_dtype)
            piece = (s.l0, s.l1, s.m0, s.m1, ref["c"])
            amax[0] = ref["amax"]
        sh.allreduce_amax(amax)
        pieces = [None] * world
        dist.all_gather_object(pieces, piece)
        if rank == 0:
            out["pieces"] = pieces
        out[rank] = float(amax[0])
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,world", [("batches", 2), ("rows", 2), ("rows", 3), ("mixed", 3),
                                        ("empty rank", 2)])
def test_sharded_result_equals_the_whole(name, world):
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(world, port, name, out), nprocs=world, join=True,
                       start_method="spawn")
    p = CASES[name]
    inp = synth.uniform_codes(p, 11, 118, 132)
    full = oracle.reference(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                            inp.SFA, inp.SFB, p.c_dtype)
    C = np.full((p.L, p.M, p.N), np.nan)
    for piece in out["pieces"]:
        if piece is not None:
            l0, l1, m0, m1, c = piece
            C[l0:l1, m0:m1] = c
    np.testing.assert_array_equal(C, full["c"])
    # every rank holds the global Amax after the one all-reduce
    assert all(out[r] == np.float32(full["amax"]) for r in range(world))
