"""Failure detection on the GPU without a fault: every pipeline wait in the
kernel is bounded.  With a wait limit far below a tile's running time the
waits run out; the kernel records it in the workspace error word, abandons
its pipeline, drains its own copies and MMAs, frees tensor memory and
returns.  The drains wait on the barriers the copies and MMAs complete on
(in a CTA pair the leader settles the stages only one CTA issued), so an
abandoned launch returns within microseconds of its first timeout, not after
a drain's own limit.  The host reads BSG_ERR_DEVICE_TIMEOUT, and the same
context then runs a normal plan correctly."""

import time

import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import synth
from gpu_util import assert_parity, problem_of, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bsg.build()
    bsg.library()


@pytest.mark.parametrize("tile_n,cluster_m", [(0, 0), (128, 1), (256, 2)],
                         ids=["default", "single-cta", "cta-pair"])
def test_wait_limit_reports_timeout_then_context_recovers(tile_n, cluster_m, monkeypatch):
    inp = synth.workload(2, M=1024, N=1024, K=4096)
    p = inp.problem
    monkeypatch.setenv("BSG_WAIT_LIMIT_NS", "2000")  # 2 us: shorter than one tile
    op = bsg.GemmAmax(problem_of(p, tile_n=tile_n, cluster_m=cluster_m))  # the plan reads the limit
    if cluster_m == 2:
        assert op.describe()["cluster_m"] == 2
    monkeypatch.delenv("BSG_WAIT_LIMIT_NS")
    A, B, SFA, SFB = to_device(inp)
    C = torch.zeros(synth.c_shape(p), dtype=torch.bfloat16, device="cuda:0")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda:0")
    op.run(A, B, SFA, SFB, C, amax)
    torch.cuda.synchronize()  # the kernel returned (no hang, no fault)
    assert op.device_status() == bsg.BSG_ERR_DEVICE_TIMEOUT
    assert op.device_status() == bsg.BSG_OK  # reading clears the error word
    # again, timed: no drain sat out its 200 ms floor
    t0 = time.perf_counter()
    op.run(A, B, SFA, SFB, C, amax)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert op.device_status() == bsg.BSG_ERR_DEVICE_TIMEOUT
    assert elapsed < 0.1, f"abandoned launch took {elapsed * 1e3:.1f} ms"
    op.close()
    # a normal plan on the same context
    c, a, *_ = run_gpu(inp, tile_n=tile_n, cluster_m=cluster_m)
    assert_parity(inp, c, a)


def test_k_halves_timeout_leaves_the_workspace_reusable(monkeypatch):
    """A plan whose leftover tiles run as K halves (the claim, the partial
    sums and the bounded wait for the claimant's flag in its epilogues),
    abandoned by the same 2 us wait limit: the launch returns with
    BSG_ERR_DEVICE_TIMEOUT, and its workspace, once the error word is read,
    serves a plan with the normal limit to parity (the abandoned launch left
    the K halves' words zero)."""
    G = bsg.GemmAmax(problem_of(synth.Problem(8192, 8192, 256, 1))).describe()["grid"] // 2
    inp = synth.workload(2, M=256 * (2 * G + 8) - 64, N=256, K=1024)
    p = inp.problem
    monkeypatch.setenv("BSG_KSPLIT_MIN_STAGES", "2")  # K halves at 8 K stages
    monkeypatch.setenv("BSG_WAIT_LIMIT_NS", "2000")
    op = bsg.GemmAmax(problem_of(p))
    monkeypatch.delenv("BSG_WAIT_LIMIT_NS")
    assert op.describe()["k_split_tiles"] == 8
    A, B, SFA, SFB = to_device(inp)
    C = torch.zeros(synth.c_shape(p), dtype=torch.bfloat16, device="cuda:0")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda:0")
    for _ in range(2):
        op.run(A, B, SFA, SFB, C, amax)
        torch.cuda.synchronize()
        assert op.device_status() == bsg.BSG_ERR_DEVICE_TIMEOUT
    assert op.device_status() == bsg.BSG_OK
    ok = bsg.GemmAmax(problem_of(p))
    assert ok.ws_bytes == op.ws_bytes and ok.describe()["k_split_tiles"] == 8
    s = torch.cuda.current_stream().cuda_stream
    C.fill_(float("nan"))
    st = bsg.bsg_run(ok.plan, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                     C.data_ptr(), amax.data_ptr(), op.workspace.data_ptr(), op.ws_bytes, s)
    assert st == bsg.BSG_OK
    torch.cuda.synchronize()
    assert bsg.bsg_check_device_status(ok.plan, op.workspace.data_ptr(), s) == bsg.BSG_OK
    c = C.float().cpu().numpy().astype("float64")
    assert_parity(inp, c, float(amax.item()))
