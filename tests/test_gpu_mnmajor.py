"""GPU parity of MN-major FP8 operands: A m-major and/or B n-major ("GEMM + Amax
(SM100)", "Parameters": A (M, K, L) with strides (1, M, M*K) for m-major, B
likewise for n-major; packed FP4 stays k-major).  The tiles land in shared
memory with the MN index contiguous and the MMA reads them transposed.  The
oracle reads the same bytes at the page's strides.  Bound as everywhere:
|C_gpu - C_ref| <= 1e-5 S + ulp_c, Amax bit-equal to max |C_gpu|."""
import numpy as np
import pytest

import block_scaled_precision_04_gb300 as bsg
import synth
from gpu_util import assert_parity, run_gpu

pytestmark = pytest.mark.gpu

MAJORS = [("m", "k"), ("k", "n"), ("m", "n")]


def P(M, N, K, L=1, am="m", bm="n", a="e4m3", b="e4m3", c="f32", major="n"):
    return synth.Problem(M, N, K, L, a, b, 32, c, major, a_major=am, b_major=bm)


SHAPES = [
    dict(M=16, N=16, K=32),                      # one MMA, mostly zero-filled tiles
    dict(M=128, N=128, K=128),
    dict(M=144, N=160, K=96, L=2),               # ragged M and N tiles, K tail
    dict(M=256, N=256, K=512),
    dict(M=400, N=528, K=224, L=3),
    dict(M=1040, N=272, K=1536),                 # ring wrap, ghost M tile of a pair
]


@pytest.mark.parametrize("am,bm", MAJORS, ids=["A-m", "B-n", "A-m_B-n"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(str(v) for v in s.values()))
def test_mn_major(am, bm, shape):
    p = P(**shape, am=am, bm=bm)
    inp = synth.uniform_codes(p, shape["M"] + 7 * shape["N"] + shape["K"] + len(am + bm), 122, 132)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096)
    assert guard_ok
    assert_parity(inp, c, amax)


@pytest.mark.parametrize("K", [40, 72, 200])
def test_k_not_a_multiple_of_16(K):
    """Both operands MN-major: nothing is contiguous along K, so any K works;
    the last K slice is partly zero-filled by the TMA."""
    p = P(272, 176, K, L=2)
    inp = synth.uniform_codes(p, K, 120, 134)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096)
    assert guard_ok
    assert_parity(inp, c, amax)


@pytest.mark.parametrize("a,b", [("e5m2", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e5m2")])
@pytest.mark.parametrize("c,major", [("bf16", "n"), ("f16", "m"), ("f32", "m")])
def test_dtypes_and_c_layouts(a, b, c, major):
    p = P(384, 320, 256, L=2, a=a, b=b, c=c, major=major)
    inp = synth.uniform_codes(p, 11 + len(a + b + c + major), 118, 126)
    c_gpu, amax, _, _, guard_ok = run_gpu(inp, guard=4096)
    assert guard_ok
    assert_parity(inp, c_gpu, amax)


@pytest.mark.parametrize("am,bm", MAJORS, ids=["A-m", "B-n", "A-m_B-n"])
@pytest.mark.parametrize("tile_n,cluster_m", [(128, 0), (224, 2), (256, 2)])
def test_tiles(am, bm, tile_n, cluster_m):
    """The 128-wide single CTA, the 224-wide pair (two accumulators, each CTA
    loading a 112-column half of B as a 128-column box) and the 256-wide pair
    (256-byte K stages)."""
    p = P(768, 1120, 1024, am=am, bm=bm, c="bf16")
    inp = synth.uniform_codes(p, tile_n + cluster_m + len(am + bm), 122, 130)
    c, amax, _, op, guard_ok = run_gpu(inp, guard=4096, tile_n=tile_n, cluster_m=cluster_m)
    assert op.describe()["tile_n"] == tile_n
    assert guard_ok
    assert_parity(inp, c, amax)


@pytest.mark.parametrize("cluster_m", [1, 2])
def test_m_major_a_with_k_major_b_clusters(cluster_m):
    """An m-major A with k-major B runs in single 256-wide CTAs and in
    256-row CTA pairs."""
    p = P(640, 768, 512, am="m", bm="k", c="bf16")
    inp = synth.uniform_codes(p, 50 + cluster_m, 122, 130)
    c, amax, _, _, guard_ok = run_gpu(inp, guard=4096, tile_n=256, cluster_m=cluster_m)
    assert guard_ok
    assert_parity(inp, c, amax)


def test_small_m_n_major_b_takes_128_wide_tiles():
    """One M tile (no pair possible): an n-major B falls back to the
    128-wide single-CTA tile."""
    p = P(96, 512, 256, am="k", bm="n")
    inp = synth.uniform_codes(p, 3, 122, 130)
    c, amax, _, op, guard_ok = run_gpu(inp, guard=4096)
    assert op.describe()["tile_n"] == 128
    assert guard_ok
    assert_parity(inp, c, amax)


def test_n_major_b_rejected_on_one_256_wide_cta():
    prob = bsg.make_problem(512, 512, 256, 1, "e4m3", "e4m3", 32, "f32", "n", b_major="n",
                            tile_n=256, cluster_m=1)
    st, _ = bsg.bsg_plan_create(prob, 0)
    assert st == bsg.BSG_ERR_UNSUPPORTED


def test_layouts_give_the_same_result():
    """The same logical operands, k-major and MN-major: the kernel's C is
    identical bit for bit (the MMAs see the same values in the same order)."""
    pk = P(512, 640, 768, am="k", bm="k", c="bf16")
    inp = synth.uniform_codes(pk, 99, 122, 130)
    ck, ak, *_ = run_gpu(inp)
    pm = P(512, 640, 768, am="m", bm="n", c="bf16")
    inm = synth.Inputs(pm, np.ascontiguousarray(inp.A.transpose(0, 2, 1)),
                       np.ascontiguousarray(inp.B.transpose(0, 2, 1)), inp.SFA, inp.SFB)
    cm, am, *_ = run_gpu(inm)
    np.testing.assert_array_equal(ck, cm)
    assert ak == am
