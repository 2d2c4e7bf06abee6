"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI on synth inputs and compare with the oracle."""
import numpy as np
import torch

import block_scaled_precision_04_gb300 as bsg
import oracle
import synth

TORCH_C = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16,
           "e4m3": torch.uint8, "e5m2": torch.uint8, "e2m1": torch.uint8}
LOW_C = ("e4m3", "e5m2", "e2m1")
POISON_BYTE = 0xA5


def problem_of(p: synth.Problem, **hints) -> bsg.bsg_problem:
    return bsg.make_problem(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, p.c_dtype,
                            p.c_major, sf_dtype=p.sf_dtype, a_major=p.a_major,
                            b_major=p.b_major, **hints)


def to_device(inp: synth.Inputs, dev="cuda:0"):
    return [torch.from_numpy(np.ascontiguousarray(x)).to(dev) for x in
            (inp.A, inp.B, inp.SFA, inp.SFB)]


def c_to_logical(c: torch.Tensor, p: synth.Problem) -> np.ndarray:
    """Device C in its memory layout -> float64 numpy (L, M, N); FP8 / E2M1
    codes are decoded with the oracle's tables."""
    if p.c_dtype in LOW_C:
        codes = c.cpu().numpy()
        if p.c_dtype == "e2m1":
            full = np.empty(codes.shape[:2] + (codes.shape[2] * 2,), dtype=np.uint8)
            full[..., 0::2] = codes & 0xF
            full[..., 1::2] = codes >> 4
            codes = full
        x = oracle.decode_table(p.c_dtype)[codes]
    else:
        x = c.float().cpu().numpy().astype(np.float64)
    return x if p.c_major == "n" else x.transpose(0, 2, 1)


def run_gpu(inp: synth.Inputs, op=None, runs=1, guard=0, **hints):
    """Launch `runs` times; returns (C logical float64, amax, raw C tensor, op, guard ok)."""
    p = inp.problem
    if op is None:
        op = bsg.GemmAmax(problem_of(p, **hints))
    A, B, SFA, SFB = to_device(inp)
    shape = synth.c_shape(p)
    numel = int(np.prod(shape))
    poison = POISON_BYTE if p.c_dtype in LOW_C else float("nan")
    buf = torch.full((numel + 2 * guard,), poison, dtype=TORCH_C[p.c_dtype], device="cuda:0")
    C = buf[guard:guard + numel].view(shape)
    amax = torch.full((1,), -1.0, dtype=torch.float32, device="cuda:0")
    for _ in range(runs):
        op.run(A, B, SFA, SFB, C, amax)
    torch.cuda.synchronize()
    st = op.device_status()
    assert st == bsg.BSG_OK, bsg.bsg_status_string(st)
    guard_ok = True
    if guard:
        g = torch.cat([buf[:guard], buf[guard + numel:]])
        guard_ok = bool((g == POISON_BYTE).all()) if p.c_dtype in LOW_C else \
            bool(torch.isnan(g.float()).all())
    return c_to_logical(C, p), float(amax.item()), C, op, guard_ok


def abs_max_bits(c: np.ndarray) -> int:
    """max |c| as float32 bit pattern (integer max, as the kernel keeps it)."""
    u = np.abs(c.astype(np.float32)).view(np.uint32)
    return int(u.max()) if u.size else 0


def assert_parity(inp: synth.Inputs, c_gpu: np.ndarray, amax_gpu: float, ref=None):
    """Elementwise |C_gpu - C_ref| <= 1e-5 * S + ulp_c(|C_ref|); Amax equal
    (bit for bit) to max |C_gpu| and within max tau of the oracle's Amax."""
    p = inp.problem
    if ref is None:
        ref = oracle.reference(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                               inp.SFA, inp.SFB, p.c_dtype, sf_dtype=p.sf_dtype,
                               a_major=p.a_major, b_major=p.b_major)
    finite = np.isfinite(ref["c"])
    with np.errstate(invalid="ignore"):
        err = np.abs(c_gpu - ref["c"])
    # where the oracle's rounded value overflows C's dtype, the stored value
    # must be that same infinity
    bad = np.where(finite, ~(err <= ref["tau"]), c_gpu != ref["c"])
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = [(tuple(int(v) for v in i), float(c_gpu[tuple(i)]), float(ref["c"][tuple(i)]),
                   float(ref["tau"][tuple(i)])) for i in idx]
        raise AssertionError(f"{int(bad.sum())} of {bad.size} elements outside tolerance; "
                             f"first (l,m,n), gpu, ref, tau: {detail}")
    assert np.float32(amax_gpu).view(np.uint32) == abs_max_bits(c_gpu), (amax_gpu, np.abs(c_gpu).max())
    if np.isfinite(ref["amax"]):
        assert abs(amax_gpu - ref["amax"]) <= float(ref["tau"][finite].max())
    else:
        assert amax_gpu == ref["amax"]
    return ref


def run_gpu_host(inp: synth.Inputs, **hints):
    """bsg_run_host: pinned host A/B/scales in, host C and Amax out (copies
    and the launch enqueued on one stream).  Returns (C logical float64, amax)."""
    p = inp.problem
    op = bsg.GemmAmax(problem_of(p, **hints))
    dA, dB, dSFA, dSFB = to_device(inp)
    shape = synth.c_shape(p)
    dC = torch.empty(shape, dtype=TORCH_C[p.c_dtype], device="cuda:0")
    damax = torch.empty(1, dtype=torch.float32, device="cuda:0")
    dev = bsg.bsg_device_buffers(dA.data_ptr(), dB.data_ptr(), dSFA.data_ptr(), dSFB.data_ptr(),
                                 dC.data_ptr(), damax.data_ptr(), op.workspace.data_ptr(),
                                 op.ws_bytes)
    hA, hB, hSFA, hSFB = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
                          for x in (inp.A, inp.B, inp.SFA, inp.SFB)]
    hC = torch.empty(shape, dtype=TORCH_C[p.c_dtype]).pin_memory()
    hamax = torch.empty(1, dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    st = bsg.bsg_run_host(op.plan, hA.data_ptr(), hB.data_ptr(), hSFA.data_ptr(),
                          hSFB.data_ptr(), hC.data_ptr(), hamax.data_ptr(), dev, s)
    assert st == bsg.BSG_OK, bsg.bsg_status_string(st)
    torch.cuda.synchronize()
    assert op.device_status() == bsg.BSG_OK
    return c_to_logical(hC, p), float(hamax[0])

