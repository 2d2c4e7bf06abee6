"""GPU parity: the CUDA path, called through the C ABI, against the oracle.

Bar ("GEMM + Amax (SM100)", section "Equations", with the tolerance the
acceptance criterion fixes): |C_gpu - C_ref| <= 1e-5 * sum_k |Ahat Bhat| +
ulp_c(|C_ref|) elementwise; Amax bit-equal to max |C_gpu| and within max tau
of the oracle's Amax.  Small shapes span several tiles and ragged tails and
are compared in full; the five workloads run at full size in the benchmark's
launch configuration and are compared at sampled points.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import oracle
import synth
from gpu_util import abs_max_bits, assert_parity, problem_of, run_gpu, run_gpu_host, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bsg.build()
    bsg.library()


def P(M, N, K, L=1, a="e4m3", b="e4m3", sfv=32, c="f32", major="n"):
    return synth.Problem(M, N, K, L, a, b, sfv, c, major)


# --------------------------------------------------------- isolated paths

def test_unit_scales_data_path():
    """Scale bytes all 127: checks the operand path (TMA, swizzle, MMA,
    epilogue) independently of the scale path."""
    inp = synth.uniform_codes(P(256, 256, 256), 21, 127, 127)
    c, amax, *_ = run_gpu(inp)
    assert_parity(inp, c, amax)


def test_scale_path_rows_and_blocks():
    """Distinct scales per (row, K-block): a wrong atom index or scale byte
    selection shows up here."""
    inp = synth.uniform_codes(P(256, 256, 512), 22, 120, 134)
    c, amax, *_ = run_gpu(inp)
    assert_parity(inp, c, amax)


def test_workload_uniform_codes_full():
    """The 256^3 uniform-code E4M3 workload, whole."""
    inp = synth.workload(1)
    c, amax, *_ = run_gpu(inp)
    assert_parity(inp, c, amax)


# ------------------------------------------------- workloads at reduced size

REDUCED = [
    (2, dict(M=640, N=512, K=1024)),
    (3, dict(M=384, N=256, K=2048, L=2)),
    (4, dict(M=512, N=384, K=1024)),
    (5, dict(M=328, N=200, K=896, L=2)),
    (6, dict(M=384, N=640, K=1024)),
    (7, dict(M=640, N=512, K=1024)),
]


@pytest.mark.parametrize("number,shape", REDUCED, ids=[f"w{n}" for n, _ in REDUCED])
def test_workload_recipe_reduced(number, shape):
    inp = synth.workload(number, **shape)
    c, amax, *_ = run_gpu(inp)
    assert_parity(inp, c, amax)


# ------------------------------------------------- ragged, tiny, variants

RAGGED = [
    P(1, 4, 32), P(127, 128, 64), P(129, 132, 96, 3), P(200, 200, 64),
    P(4, 1, 32, 2, major="m"), P(128, 127, 96, major="m"), P(132, 129, 64, 3, major="m"),
    P(200, 72, 48), P(72, 200, 112, 2, c="bf16"), P(130, 136, 208, c="f16"),
    P(257, 264, 160, a="e5m2", b="e5m2"), P(96, 160, 64, a="e4m3", b="e5m2", major="m"),
]


@pytest.mark.parametrize("p", RAGGED, ids=[f"{p.M}x{p.N}x{p.K}L{p.L}{p.c_major}{p.c_dtype}{p.a_dtype}{p.b_dtype}" for p in RAGGED])
def test_ragged_shapes(p):
    lo, hi = (118, 124) if p.c_dtype == "f16" else (122, 132)  # keep most of fp16 finite
    inp = synth.uniform_codes(p, p.M * 7 + p.N * 3 + p.K, lo, hi)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096)
    assert guard_ok, "write outside C"
    assert_parity(inp, c, amax)


FP4 = [
    P(128, 128, 64, a="e2m1", b="e2m1", sfv=16),
    P(200, 136, 96, 2, a="e2m1", b="e2m1", sfv=16, c="bf16"),
    P(256, 128, 512, a="e2m1", b="e2m1", sfv=32),
    P(132, 200, 160, a="e2m1", b="e2m1", sfv=32, major="m"),
    P(129, 128, 32, a="e2m1", b="e2m1", sfv=16, c="f16"),
]


@pytest.mark.parametrize("p", FP4, ids=[f"{p.M}x{p.N}x{p.K}L{p.L}sfv{p.sfv}{p.c_major}{p.c_dtype}" for p in FP4])
def test_fp4(p):
    inp = synth.uniform_codes(p, p.M + p.N + p.K + p.sfv, 123, 131)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096)
    assert guard_ok
    assert_parity(inp, c, amax)


def test_amax_overwritten_not_accumulated():
    """Amax is per run: a second run with smaller values reports its own max."""
    big = synth.uniform_codes(P(256, 128, 128), 31, 130, 130)
    small = synth.uniform_codes(P(256, 128, 128), 32, 120, 120)
    c1, a1, _, op, _ = run_gpu(big)
    c2, a2, *_ = run_gpu(small, op=op)
    assert a1 > a2
    assert np.float32(a2).view(np.uint32) == abs_max_bits(c2)
    assert_parity(small, c2, a2)


def test_repeated_runs_identical():
    inp = synth.workload(2, M=256, N=384, K=512)
    c1, a1, _, op, _ = run_gpu(inp, runs=3)
    c2, a2, *_ = run_gpu(inp, op=op, runs=1)
    np.testing.assert_array_equal(c1, c2)
    assert a1 == a2


def test_amax_with_nan_scale():
    """A 0xFF scale byte (E8M0 NaN) in a used block of row 5: the other rows
    are unaffected and Amax is still the integer max of the stored bits."""
    inp = synth.uniform_codes(P(128, 128, 64), 33, 127, 127)
    sfa = inp.SFA.copy()
    sfa[0, 0, 0, 5, 0, 0] = 0xFF  # row 5, K-block 0
    inp = synth.Inputs(inp.problem, inp.A, inp.B, sfa, inp.SFB)
    c, amax, *_ = run_gpu(inp)
    assert np.float32(amax).view(np.uint32) == abs_max_bits(c)
    p = inp.problem
    ref = oracle.reference(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                           inp.SFA, inp.SFB, p.c_dtype)
    keep = np.arange(p.M) != 5
    assert np.all(np.abs(c[:, keep] - ref["c"][:, keep]) <= ref["tau"][:, keep])


def test_run_validation_statuses():
    inp = synth.uniform_codes(P(128, 128, 64), 34, 127, 127)
    op = bsg.GemmAmax(problem_of(inp.problem))
    A, B, SFA, SFB = to_device(inp)
    C = torch.empty((1, 128, 128), dtype=torch.float32, device="cuda:0")
    amax = torch.empty(1, dtype=torch.float32, device="cuda:0")
    s = torch.cuda.current_stream().cuda_stream
    ws = op.workspace.data_ptr()
    run = lambda **kw: bsg.bsg_run(op.plan, kw.get("A", A.data_ptr()), B.data_ptr(),
                                   SFA.data_ptr(), SFB.data_ptr(), kw.get("C", C.data_ptr()),
                                   amax.data_ptr(), kw.get("ws", ws), kw.get("wsb", op.ws_bytes), s)
    assert run(A=A.data_ptr() + 8) == bsg.BSG_ERR_ALIGNMENT
    assert run(C=C.data_ptr() + 4) == bsg.BSG_ERR_ALIGNMENT
    assert run(wsb=op.ws_bytes - 1) == bsg.BSG_ERR_WORKSPACE
    assert run(ws=0) == bsg.BSG_ERR_WORKSPACE
    assert run(A=0) == bsg.BSG_ERR_INVALID_ARG
    assert run() == bsg.BSG_OK
    torch.cuda.synchronize()
    assert op.device_status() == bsg.BSG_OK


def test_plan_describe():
    op = bsg.GemmAmax(bsg.make_problem(4096, 4096, 4096, 1, c_dtype="bf16"))
    info = op.describe()
    assert info["tile_m"] == 128 and info["stages"] >= 2
    assert info["grid"] == min(info["num_tiles"], torch.cuda.get_device_properties(0).multi_processor_count)
    assert info["kernel_name"]


HOST_CASES = [
    P(256, 256, 256, c="bf16"),
    P(300, 224, 384, 2, a="e2m1", b="e2m1", sfv=16, c="e2m1"),        # packed FP4 C
    P(144, 160, 256, a="e2m1", b="e2m1", sfv=16, c="e4m3", major="m"),  # FP8 C, m-major
    synth.Problem(272, 176, 96, 2, "e4m3", "e5m2", 32, "f32", "n", a_major="m", b_major="n"),
    synth.Problem(256, 384, 512, 1, "e2m1", "e2m1", 16, "bf16", "n", sf_dtype="e4m3"),
]


@pytest.mark.parametrize("p", HOST_CASES, ids=lambda p: p.describe().replace(" ", "_"))
def test_run_host_end_to_end(p):
    """bsg_run_host: host buffers in, host C and Amax out; the copies are
    sized from the problem (packed E2M1 C, MN-major operands, E4M3 scales)."""
    lo, hi = (0x30, 0x40) if p.sf_dtype == "e4m3" else (120, 128)
    inp = synth.uniform_codes(p, p.M + p.N + p.K, lo, hi)
    c, amax = run_gpu_host(inp)
    assert_parity(inp, c, amax)


# ------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("number", [1, 2, 3, 4, 5, 6, 7])
def test_workload_full_size(number):
    """Each workload at its full size, in the benchmark's launch
    configuration, against the whole oracle: every element of C within
    tau = 1e-5 * sum_k |Ahat Bhat| + ulp_c(|C_ref|), Amax bit-equal to
    max |C_gpu| and within max tau of the oracle's Amax.  (The oracle runs
    over all host cores; 8192^3 FP4 takes about half a minute.)"""
    inp = synth.workload(number)
    c, amax, _, op, _ = run_gpu(inp)
    assert_parity(inp, c, amax)


# ------------------------------------------------- tile-shape variants

TILE_CASES = [
    P(256, 512, 512), P(200, 520, 160, 2, c="bf16"), P(136, 1000, 96, major="m"),
    P(640, 1352, 1024, c="bf16"), P(392, 904, 512, 2, major="m"),
    P(1000, 1576, 384, a="e5m2", b="e4m3", c="f16"),
    P(128, 264, 64, a="e2m1", b="e2m1", sfv=16),
    P(260, 384, 640, a="e2m1", b="e2m1", sfv=16, c="bf16"),
    P(132, 392, 384, 2, a="e2m1", b="e2m1", sfv=32, major="m"),
    P(384, 1100, 256, a="e5m2", b="e4m3"),
]


@pytest.mark.parametrize("tile_n", [128, 224, 256])
@pytest.mark.parametrize("p", TILE_CASES, ids=[f"{p.M}x{p.N}x{p.K}L{p.L}{p.a_dtype}sfv{p.sfv}{p.c_major}" for p in TILE_CASES])
def test_tile_variants(p, tile_n):
    """Every tile width against the oracle, ragged N included.  256 reads two
    128-row scale groups of B per K-chunk; 224 (FP8 pairs, two accumulators)
    starts each tile at a multiple of 32 inside a scale atom, so its scales
    are gathered across up to three atoms."""
    if tile_n == 224 and (p.a_dtype == "e2m1" or p.M <= 128):
        st, _ = bsg.bsg_plan_create(problem_of(p, tile_n=224), 0)
        assert st == bsg.BSG_ERR_UNSUPPORTED
        return
    inp = synth.uniform_codes(p, p.M * 5 + p.N + p.K + tile_n, 123, 131)
    c, amax, _, op, guard_ok = run_gpu(inp, guard=4096, tile_n=tile_n)
    assert op.describe()["tile_n"] == tile_n
    assert guard_ok
    assert_parity(inp, c, amax)


CLUSTER_CASES = [
    P(640, 512, 512), P(200, 520, 160, 2, c="bf16"), P(392, 1000, 96, major="m"),
    P(260, 384, 640, a="e2m1", b="e2m1", sfv=16, c="bf16"),
    P(132, 392, 384, 2, a="e2m1", b="e2m1", sfv=32, major="m"),
    P(1000, 264, 256, 3, a="e5m2", b="e4m3"),
    # more units than resident clusters and more K stages than the smem ring:
    # the ring and the accumulator hand-off wrap
    P(2048, 2560, 1024, c="bf16"),
    P(1536, 2304, 2048, a="e2m1", b="e2m1", sfv=16, c="bf16"),
]


@pytest.mark.parametrize("cluster_m", [1, 2])
@pytest.mark.parametrize("p", CLUSTER_CASES, ids=[f"{p.M}x{p.N}x{p.K}L{p.L}{p.a_dtype}sfv{p.sfv}{p.c_major}" for p in CLUSTER_CASES])
def test_cluster_shapes(p, cluster_m):
    """Single CTAs (cluster 1) or a cta_group::2 pair (cluster 2, the
    default: 256-row MMAs, each CTA holding half the B tile); M-tile counts
    that do not divide by two give a ghost tile in the last pair."""
    inp = synth.uniform_codes(p, p.M * 3 + p.N + p.K + cluster_m, 123, 131)
    c, amax, _, op, guard_ok = run_gpu(inp, guard=4096, tile_n=256, cluster_m=cluster_m)
    info = op.describe()
    assert info["tile_n"] == 256 and info["cluster_m"] >= 1
    assert guard_ok
    assert_parity(inp, c, amax)
