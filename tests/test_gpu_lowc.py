"""GPU parity of low-precision C -- E4M3, E5M2 and packed E2M1 -- from the
FP4 GEMM ("GEMM + Amax (SM100)", "Parameters": C may be float8_e4m3fn,
float8_e5m2 or float4_e2m1fn_x2; "Support surface": FP8 C with FP8 operands
is disabled, FP4 C needs FP4 operands and an n-major C).  C is the fp32
result rounded to nearest even with saturation; the oracle rounds its double
sum the same way and the per-element bound |C_gpu - C_ref| <= 1e-5 S + ulp_c
(one step of the output format) covers a sum that lands on the other side of
a rounding boundary.  Amax is max |stored C|, bit for bit."""
import pytest

import block_scaled_precision_04_gb300 as bsg
import synth
from gpu_util import assert_parity, run_gpu

pytestmark = pytest.mark.gpu


def P(M, N, K, L=1, sfv=16, c="e4m3", major="n"):
    return synth.Problem(M, N, K, L, "e2m1", "e2m1", sfv, c, major)


CASES = [
    P(256, 256, 256, c="e4m3"),
    P(256, 256, 512, c="e5m2", sfv=32),
    P(256, 256, 256, c="e2m1"),
    P(300, 224, 384, L=2, c="e4m3"),          # ragged M, N
    P(300, 224, 384, L=2, c="e2m1", sfv=32),
    P(144, 160, 256, c="e4m3", major="m"),     # m-major FP8 (rows of M bytes: M % 16 == 0)
    P(144, 160, 256, c="e5m2", major="m", sfv=32),
    P(128, 64, 128, c="e2m1"),                 # N <= 128: the 128-wide tile
    P(128, 48, 128, c="e4m3"),
]


@pytest.mark.parametrize("p", CASES, ids=lambda p: f"{p.M}x{p.N}x{p.K}x{p.L}-sfv{p.sfv}-{p.c_dtype}-{p.c_major}")
@pytest.mark.parametrize("scale_lo,scale_hi", [(118, 124), (125, 131)])
def test_low_precision_c(p, scale_lo, scale_hi):
    """Small scales keep C inside the formats' ranges (rounding exercised);
    larger ones push much of it past the largest value (saturation)."""
    inp = synth.uniform_codes(p, p.M + 3 * p.N + p.K + scale_lo, scale_lo, scale_hi)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096)
    assert guard_ok
    assert_parity(inp, c, amax)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("cdt", ["e4m3", "e2m1"])
def test_low_precision_c_tiles(tile_n, cdt):
    p = P(384, 512, 256, c=cdt)
    inp = synth.uniform_codes(p, 700 + tile_n, 120, 128)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096, tile_n=tile_n)
    assert guard_ok
    assert_parity(inp, c, amax)


def test_fp8_operands_with_fp8_c_rejected():
    prob = bsg.make_problem(128, 128, 128, 1, "e4m3", "e4m3", 32, "e4m3")
    st, _ = bsg.bsg_plan_create(prob, 0)
    assert st == bsg.BSG_ERR_UNSUPPORTED
