"""bsg_run_noalloc: the entry point for callers that cannot allocate device
memory (no allocator of their own, or code running where cudaMalloc is not
allowed).  Its workspace is a fixed array inside the library, so its
results must match bsg_run with a caller-allocated workspace, call after
call: the array keeps the previous call's contents, and two different
problems in a row show whether the entry point clears what must start at
zero.  Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import synth
from gpu_util import TORCH_C, abs_max_bits, assert_parity, problem_of, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bsg.build()
    bsg.library()


def _run_both(inp):
    p = inp.problem
    op = bsg.GemmAmax(problem_of(p))
    A, B, SFA, SFB = to_device(inp)
    shape = synth.c_shape(p)
    c_ref = torch.full(shape, float("nan"), dtype=TORCH_C[p.c_dtype], device="cuda:0")
    c_new = torch.full(shape, float("nan"), dtype=TORCH_C[p.c_dtype], device="cuda:0")
    a_ref = torch.full((1,), -1.0, device="cuda:0")
    a_new = torch.full((1,), -1.0, device="cuda:0")
    s = torch.cuda.current_stream().cuda_stream
    op.run(A, B, SFA, SFB, c_ref, a_ref)
    # the reference launch's own workspace: its pipeline waits all completed
    assert op.device_status() == bsg.BSG_OK
    st = bsg.bsg_run_noalloc(op.plan, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                             c_new.data_ptr(), a_new.data_ptr(), s)
    assert st == bsg.BSG_OK, bsg.bsg_status_string(st)
    torch.cuda.synchronize()
    return c_ref, a_ref, c_new, a_new


def _logical(c, p):
    x = c.float().cpu().numpy().astype(np.float64)
    return x if p.c_major == "n" else x.transpose(0, 2, 1)


def test_noalloc_matches_bsg_run_twice():
    """Two calls in a row (a large Amax, then a small one, different shapes
    and dtypes): each equals bsg_run on the same inputs and meets the
    oracle tolerance; the second Amax is its own, not the first's."""
    first = synth.uniform_codes(synth.Problem(256, 384, 256, 2, "e4m3", "e4m3", 32, "f32", "n"),
                                901, 128, 132)
    second = synth.workload(2, M=384, N=256, K=512)  # bf16 C, quantised N(0,1) values
    amaxes = []
    for inp in (first, second):
        p = inp.problem
        c_ref, a_ref, c_new, a_new = _run_both(inp)
        assert torch.equal(c_new.view(torch.uint8), c_ref.view(torch.uint8))
        assert a_new.item() == a_ref.item()
        c = _logical(c_new, p)
        assert np.float32(a_new.item()).view(np.uint32) == abs_max_bits(c)
        assert_parity(inp, c, float(a_new.item()))
        amaxes.append(a_new.item())
    assert amaxes[1] < amaxes[0]


def test_noalloc_rejects_bad_arguments():
    p = synth.Problem(128, 128, 64, 1)
    op = bsg.GemmAmax(problem_of(p))
    assert bsg.bsg_run_noalloc(None, 1, 1, 1, 1, 1, 1, 0) == bsg.BSG_ERR_INVALID_ARG
    assert bsg.bsg_run_noalloc(op.plan, 0, 16, 16, 16, 16, 16, 0) == bsg.BSG_ERR_INVALID_ARG
    # checked before the array is touched: a misaligned pointer enqueues nothing
    assert bsg.bsg_run_noalloc(op.plan, 8, 16, 16, 16, 16, 16, 0) == bsg.BSG_ERR_ALIGNMENT
