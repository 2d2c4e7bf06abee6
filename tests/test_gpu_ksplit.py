"""K halves of the leftover tiles: when the 256 x 256 tiles left after at
least two whole waves fill at most half of the resident CTA pairs (FP8
operands), each runs as two units over the first and the second half of the
K stages, at full width.  The half that claims the tile first writes its
fp32 partial sum to the workspace; the other adds it to its own accumulator
as it drains.  These cases check, through the C ABI: when the plan uses
them; that C and Amax stay within the oracle's tolerance on every C path of
the FP8 kernel (bf16, f16 and fp32; n- and m-major C; MN-major operands;
ragged M, N and K; odd K-stage counts); that C does not depend on which
half claims first (the halves start together, as the first units of two
clusters); that a run leaves the counters zero for the next; and that a
workspace too small for the partial sums runs the half-width split within
the same tolerance."""
import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import synth
from gpu_util import TORCH_C, assert_parity, problem_of, run_gpu, to_device

pytestmark = pytest.mark.gpu

WS_WORDS = 256  # bytes of the words every run needs; the counters follow


def P(M, N, K, L=1, a="e4m3", b="e4m3", c="f32", major="n", am="k", bm="k"):
    return synth.Problem(M, N, K, L, a, b, 32, c, major, "ue8m0", am, bm)


@pytest.fixture(scope="module", autouse=True)
def _k_halves_from_two_stages():
    """Plans made in this file take K halves from 2 K stages on (the default
    threshold, 40, would need far larger test problems)."""
    mp = pytest.MonkeyPatch()
    mp.setenv("BSG_KSPLIT_MIN_STAGES", "2")
    yield
    mp.undo()


@pytest.fixture(scope="module")
def G():
    """Resident 256-wide FP8 pairs: a full-wave problem's grid / 2."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    op = bsg.GemmAmax(problem_of(P(4096 * 2, 4096 * 2, 256)))
    return op.describe()["grid"] // 2


def with_tiles(G, extra, N, K, L=1, trim=37, **kw):
    """A problem of 2G + r tiles of 256 x 256 (r >= extra, the smallest that
    fills whole rows of N tiles in every batch) with a ragged last M tile."""
    nt = -(-N // 256)
    r = extra
    while (2 * G + r) % (nt * L):
        r += 1
    assert r <= G // 2
    mt = (2 * G + r) // (nt * L)
    return P(256 * mt - trim, N, K, L, **kw), r


# (extra tiles, N, K, L, trim, keywords): bf16 with 3 K stages (halves of 1
# and 2), fp32 m-major over two batches, f16 at the most split tiles with 2
# stages, MN-major A and B, E5M2 x E4M3 with a ragged K (8 stages, the last
# partial), fp32 n-major over four N tiles with a ragged N edge, bf16 m-major
# with a ragged N edge
SHAPES = [
    (10, 200, 384, 1, 37, dict(c="bf16")),
    (10, 256, 512, 2, 36, dict(c="f32", major="m")),
    (None, 192, 256, 1, 37, dict(c="f16")),
    (7, 256, 512, 1, 48, dict(c="bf16", am="m", bm="n")),
    (20, 160, 1008, 1, 5, dict(a="e5m2", c="f32")),
    (12, 1000, 256, 1, 100, dict(c="f32")),
    (9, 232, 512, 1, 40, dict(c="bf16", major="m")),
]
IDS = ["bf16_k3", "f32_mmajor_L2", "f16_max_split_k2", "bf16_mn_major", "e5m2_f32_ragged_k",
       "f32_ragged_n", "bf16_mmajor_ragged_n"]


def case(G, i):
    extra, N, K, L, trim, kw = SHAPES[i]
    return with_tiles(G, G // 2 if extra is None else extra, N, K, L, trim, **kw)


def inputs(p, seed):
    return synth.uniform_codes(p, seed, 123, 131)


def counters_zero(op, r):
    w = op.workspace[WS_WORDS:WS_WORDS + 16 * r].cpu().numpy()
    return bool((w == 0).all())


@pytest.mark.parametrize("i", range(len(SHAPES)), ids=IDS)
def test_k_halves_parity(G, i):
    p, r = case(G, i)
    inp = inputs(p, 300 + i)
    c, amax, _, op, guard_ok = run_gpu(inp, guard=4096)
    info = op.describe()
    assert info["k_split_tiles"] == r and info["tile_n"] == 256 and info["cluster_m"] == 2, info
    assert guard_ok, "write outside C"
    assert_parity(inp, c, amax)
    assert counters_zero(op, r)
    # a second launch on the same workspace: the counters were left zero
    c2, amax2, *_ = run_gpu(inp, op=op)
    np.testing.assert_array_equal(c2, c)
    assert amax2 == amax and counters_zero(op, r)


@pytest.mark.parametrize("i", [0, 1], ids=IDS[:2])
def test_claim_order_does_not_change_c(G, i):
    """The two halves of a split tile start together (the first units of
    two clusters), so either may claim it first, launch by launch; C and
    Amax are the same bits every time, and the counters are left zero."""
    p, r = case(G, i)
    inp = inputs(p, 400 + i)
    c1, a1, _, op, _ = run_gpu(inp)
    for _ in range(4):
        c2, a2, *_ = run_gpu(inp, op=op)
        np.testing.assert_array_equal(c2, c1)
        assert a2 == a1 and counters_zero(op, r)


def test_small_workspace_runs_half_width(G):
    """bsg_run with the 256-byte workspace every run needs: the half-width
    split of the last wave instead of the K halves, within tolerance; and
    bsg_run_noalloc (a 4096-byte array) the same."""
    p, r = case(G, 0)
    inp = inputs(p, 500)
    op = bsg.GemmAmax(problem_of(p))
    assert op.ws_bytes >= WS_WORDS + 16 * r + r * 4 * 128 * 256 * 4
    info = op.describe()
    assert info["k_split_tiles"] == r and info["half_tiles"] == r
    A, B, SFA, SFB = to_device(inp)
    shape = synth.c_shape(p)
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(WS_WORDS, dtype=torch.uint8, device="cuda:0")
    assert bsg.bsg_workspace_init(op.plan, ws.data_ptr(), WS_WORDS, s) == bsg.BSG_OK
    ref = None
    for noalloc in (False, True):
        C = torch.full(shape, float("nan"), dtype=TORCH_C[p.c_dtype], device="cuda:0")
        amax = torch.full((1,), -1.0, device="cuda:0")
        if noalloc:
            st = bsg.bsg_run_noalloc(op.plan, A.data_ptr(), B.data_ptr(), SFA.data_ptr(),
                                     SFB.data_ptr(), C.data_ptr(), amax.data_ptr(), s)
        else:
            st = bsg.bsg_run(op.plan, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                             C.data_ptr(), amax.data_ptr(), ws.data_ptr(), WS_WORDS, s)
        assert st == bsg.BSG_OK, bsg.bsg_status_string(st)
        torch.cuda.synchronize()
        if not noalloc:
            assert bsg.bsg_check_device_status(op.plan, ws.data_ptr(), s) == bsg.BSG_OK
        x = C.float().cpu().numpy().astype(np.float64)
        ref = assert_parity(inp, x, float(amax.item()), ref=ref)


def test_default_threshold_is_forty_k_stages(G, monkeypatch):
    """Without the environment setting, a plan takes K halves only from 40
    K stages (5120 FP8 bytes per row) on."""
    monkeypatch.delenv("BSG_KSPLIT_MIN_STAGES")
    short = with_tiles(G, 10, 256, 39 * 128)[0]
    long_ = with_tiles(G, 10, 256, 40 * 128)[0]
    assert bsg.GemmAmax(problem_of(short)).describe()["k_split_tiles"] == 0
    assert bsg.GemmAmax(problem_of(long_)).describe()["k_split_tiles"] > 0


@pytest.mark.parametrize("name,prob,hints", [
    ("one_whole_wave", lambda G: P(256 * (G + 5), 256, 512), {}),
    ("too_many_left", lambda G: P(256 * (2 * G + G // 2 + 1), 256, 512), {}),
    ("one_k_stage", lambda G: with_tiles(G, 10, 256, 128)[0], {}),
    ("fp4", lambda G: with_tiles(G, 10, 256, 512, a="e2m1", b="e2m1", c="bf16")[0], {}),
    ("single_ctas", lambda G: with_tiles(G, 10, 256, 512)[0], dict(tile_n=256, cluster_m=1)),
])
def test_plans_without_k_halves(G, name, prob, hints):
    p = prob(G)
    op = bsg.GemmAmax(problem_of(p, **hints))
    assert op.describe()["k_split_tiles"] == 0, (name, op.describe())
    assert op.ws_bytes == WS_WORDS
