"""GPU parity of the NVFP4 form: packed E2M1 operands with one E4M3 scale per
16 elements ("GEMM + Amax (SM100)", "Parameters": SFA/SFB may be
float8_e4m3fn; "Dtypes": E4M3 scales only with sf_vec_size 16, and sfv 16
only with FP4 operands).  The scales are unsigned E4M3 (sign bit clear): the
tensor cores read them as UE4M3, the oracle decodes the byte as float8_e4m3fn.
Same bound as every other parity test: |C_gpu - C_ref| <= 1e-5 S + ulp_c, Amax
bit-equal to max |C_gpu|."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from gpu_util import abs_max_bits, assert_parity, run_gpu

pytestmark = pytest.mark.gpu


def P(M, N, K, L=1, c="f32", major="n"):
    return synth.Problem(M, N, K, L, "e2m1", "e2m1", 16, c, major, sf_dtype="e4m3")


CASES = [
    P(128, 128, 64),
    P(256, 256, 256, c="bf16"),
    P(300, 224, 416, L=2),                    # ragged M, N; K of 26 blocks (ragged atom)
    P(1, 16, 32),                             # one row, one K step
    P(136, 1000, 96, major="m"),              # m-major C
    P(260, 384, 640, c="f16"),
    P(256, 256, 256, c="e4m3"),               # low-precision C
    P(300, 224, 384, L=2, c="e2m1"),
    P(144, 160, 256, c="e5m2", major="m"),
]

# E4M3 scale-byte ranges: around 1.0; small normals down into the subnormals;
# the top of the format (up to 448).
SCALES = [(0x30, 0x40), (0x01, 0x12), (0x68, 0x7E)]


@pytest.mark.parametrize("p", CASES, ids=lambda p: f"{p.M}x{p.N}x{p.K}x{p.L}-{p.c_dtype}-{p.c_major}")
@pytest.mark.parametrize("lo,hi", SCALES, ids=["unit", "subnormal", "top"])
def test_e4m3_scales(p, lo, hi):
    if p.c_dtype in ("e4m3", "e5m2", "e2m1") and lo == 0x68:
        lo, hi = 0x48, 0x58  # keep some of C inside the narrow output formats
    if p.c_dtype == "f16" and lo == 0x68:
        lo, hi = 0x40, 0x48  # no sums near fp16's overflow threshold
    inp = synth.uniform_codes(p, 31 * p.M + p.N + p.K + lo, lo, hi)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096)
    assert guard_ok
    assert_parity(inp, c, amax)


@pytest.mark.parametrize("tile_n,cluster_m", [(128, 0), (256, 1), (256, 2)])
def test_e4m3_scales_tiles(tile_n, cluster_m):
    """Every tile width and cluster shape of the FP4 kernel, with the pipeline
    ring and the accumulator hand-off wrapping."""
    p = P(1536, 2304, 2048, c="bf16")
    inp = synth.uniform_codes(p, 900 + tile_n + cluster_m, 0x2C, 0x44)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096, tile_n=tile_n, cluster_m=cluster_m)
    assert guard_ok
    assert_parity(inp, c, amax)


def test_e4m3_scale_is_not_read_as_e8m0():
    """One scale byte 0x38 (E4M3 1.0) everywhere: C equals the plain product
    of the codes; read as E8M0 it would be 2^-142 times that."""
    p = P(128, 128, 128)
    inp = synth.uniform_codes(p, 4, 0x38, 0x38)
    c, amax, *_ = run_gpu(inp)
    ref = oracle.reference(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                           inp.SFA, inp.SFB, p.c_dtype, sf_dtype="e4m3")
    np.testing.assert_array_equal(c, ref["c"])  # small integers times halves: exact in fp32


def test_e4m3_scales_full_size_sampled():
    """8192^3 NVFP4 with E4M3 scales (the FP4 workload's shape and launch
    configuration): the oracle at 4096 seeded points plus the corners and
    the GPU's argmax; Amax bit-equal to max |C_gpu|."""
    p = dataclasses.replace(synth.WORKLOADS[4][1], sf_dtype="e4m3")
    inp = synth.uniform_codes(p, 4242, 0x28, 0x40)
    c, amax, *_ = run_gpu(inp)
    assert np.float32(amax).view(np.uint32) == abs_max_bits(c)
    arg = np.unravel_index(np.argmax(np.abs(c)), c.shape)
    extra = [(arg[1], arg[2], arg[0]), (p.M - 1, p.N - 1, p.L - 1), (0, 0, 0)]
    pts = synth.sample_points(p, 4096, 4243, extra)
    cref, s = oracle.gemm_sample(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A,
                                 inp.B, inp.SFA, inp.SFB, pts, sf_dtype="e4m3")
    cref = oracle.round_to(cref, p.c_dtype)
    tau = oracle.tolerance(cref, s, p.c_dtype)
    got = c[pts[:, 2], pts[:, 0], pts[:, 1]]
    bad = ~(np.abs(got - cref) <= tau)
    assert not bad.any(), [(tuple(pts[i]), got[i], cref[i]) for i in np.flatnonzero(bad)[:8]]
