"""The split last wave: when the 256 x 256 tiles left after the full waves
fill at most half of the resident CTA pairs, each runs as two 256 x 128
half-width units (N = 128 MMAs, 64 rows of B per CTA, half the epilogue
columns per warp).  These cases check, through the C ABI, that the plan
splits exactly when it should and that C and Amax stay within the oracle's
tolerance when whole tiles and halves share one launch, at ragged N and M
edges, for every C path (fp32 n- and m-major, bf16, FP8 C from FP4
operands) and both FP8 and FP4 kernels."""
import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import synth
from gpu_util import assert_parity, problem_of, run_gpu

pytestmark = pytest.mark.gpu


def P(M, N, K, L=1, a="e4m3", b="e4m3", sfv=32, c="f32", major="n", sf="ue8m0", am="k",
      bm="k"):
    return synth.Problem(M, N, K, L, a, b, sfv, c, major, sf, am, bm)


def pairs_resident() -> int:
    """Resident 256-wide FP8 pairs: a full-wave problem's grid / 2."""
    op = bsg.GemmAmax(problem_of(P(4096 * 2, 4096 * 2, 256)))
    return op.describe()["grid"] // 2


def expected_half_tiles(units: int, G: int) -> int:
    tail = units % G
    return tail if tail and 2 * tail <= G else 0


@pytest.mark.parametrize("M,N,L", [(4096, 4096, 1), (512, 768, 1), (512, 256 * 43, 1),
                                   (2048, 2048, 8), (1000, 1000, 2), (256, 256, 1)])
def test_plan_splits_the_last_wave(M, N, L):
    """half_tiles = the tiles past the full waves, when they fill at most
    half of the resident pairs; else none."""
    G = pairs_resident()
    op = bsg.GemmAmax(problem_of(P(M, N, 512, L), tile_n=256))
    info = op.describe()
    units = -(-M // 256) * -(-N // 256) * L
    assert info["tile_n"] == 256 and info["cluster_m"] == 2
    assert info["half_tiles"] == expected_half_tiles(units, G), (units, G, info)


def test_small_problems_take_128_wide_single_ctas():
    """With no hints, a problem whose 128 x 128 tiles fill at most half of
    the SMs runs as 128-wide single CTAs (latency-bound work); a larger one
    as 256-wide pairs."""
    op = bsg.GemmAmax(problem_of(P(256, 256, 256)))
    info = op.describe()
    assert info["tile_n"] == 128 and info["cluster_m"] == 1
    op = bsg.GemmAmax(problem_of(P(4096, 4096, 512)))
    info = op.describe()
    assert info["tile_n"] == 256 and info["cluster_m"] == 2


def test_no_split_for_single_ctas_or_n_major_b():
    op = bsg.GemmAmax(problem_of(P(512, 768, 256), tile_n=256, cluster_m=1))
    assert op.describe()["half_tiles"] == 0
    op = bsg.GemmAmax(problem_of(P(512, 768, 256, bm="n"), tile_n=256, cluster_m=2))
    assert op.describe()["half_tiles"] == 0


CASES = [
    # whole tiles and halves in one launch: 86 units -> 76 whole + 20 halves
    P(512, 256 * 43, 256, c="bf16"),
    # every unit a half; ragged N edge (1000 = 3 * 256 + 232) inside the last
    # tile's second half, ragged M (a ghost row block) and two batches
    P(1000, 1000, 512, 2),
    P(1000, 1000, 512, 2, major="m"),
    P(1000, 1000, 512, 2, c="bf16", major="m"),
    P(640, 1000, 320, 1, a="e5m2", b="e4m3", c="f16"),
    # FP4 kernels: MXFP4 (sfv 32), NVFP4 (E4M3 scales), FP8 C
    P(768, 1280, 512, 1, a="e2m1", b="e2m1", sfv=32, c="bf16"),
    P(768, 1280, 512, 1, a="e2m1", b="e2m1", sfv=16, c="f32", sf="e4m3"),
    P(768, 1280, 512, 1, a="e2m1", b="e2m1", sfv=16, c="e4m3"),
    P(768, 1280, 512, 1, a="e2m1", b="e2m1", sfv=16, c="e2m1"),
    # m-major A (k-major B): halves allowed
    P(512, 768, 384, 1, am="m", c="bf16"),
]


@pytest.mark.parametrize("p", CASES, ids=[f"{p.M}x{p.N}x{p.K}L{p.L}{p.a_dtype}{p.sf_dtype}sfv{p.sfv}"
                                          f"{p.c_dtype}{p.c_major}{p.a_major}" for p in CASES])
def test_split_parity(p):
    inp = synth.uniform_codes(p, p.M + p.N + p.K + p.L, 123, 131) if p.sf_dtype == "ue8m0" \
        else synth.uniform_codes(p, p.M + p.N + p.K + p.L, 0x2C, 0x44)
    c, amax, _, op, guard_ok = run_gpu(inp, guard=4096, tile_n=256)
    assert op.describe()["half_tiles"] > 0
    assert guard_ok, "write outside C"
    assert_parity(inp, c, amax)


def test_split_matches_the_unsplit_single_cta_plan():
    """The same problem through the split pair plan and through single
    256-wide CTAs (no split): both within tolerance of the oracle, and their
    Amax each equal to max |C| of their own C."""
    p = P(512, 256 * 43, 256, c="f32")
    inp = synth.uniform_codes(p, 77, 123, 131)
    c1, a1, _, op1, _ = run_gpu(inp, tile_n=256)
    c2, a2, _, op2, _ = run_gpu(inp, tile_n=256, cluster_m=1)
    assert op1.describe()["half_tiles"] > 0 and op2.describe()["half_tiles"] == 0
    ref = assert_parity(inp, c1, a1)
    assert_parity(inp, c2, a2, ref=ref)
