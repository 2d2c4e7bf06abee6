"""Block-scaled (MX) batched GEMM + global Amax on GB300 (sm_103a).

Python binding of ``libbsgemm.so``, the C ABI declared in ``include/bsgemm.h``.
Argument marshalling only: every step of the operation runs in the CUDA
library; there is no Python or CPU fallback.  Any call raises ``RuntimeError``
when the library has not been built (``build()`` or ``__graft_entry__.build()``).

Operation ("GEMM + Amax (SM100)", section "Equations"): for A (M,K,L) and
B (N,K,L) holding FP8 or packed FP4 codes with E8M0 scales per sf_vec_size
K-block in the 128-row atom layout, C[m,n,l] = sum_k Ahat[m,k,l] Bhat[n,k,l]
and Amax = max |C|.

The MX quantizer that produces such operands ("GEMM + RoPE + MXFP8
Projection (SM100)", section "Equations"; ``include/bsquant.h``) is bound here
too: ``bsg_quant_check``, ``bsg_quant_sizes``, ``bsg_quantize`` and the torch
convenience ``quantize``.

The functions keep the C names and return the C status code (0 = BSG_OK);
functions with C out-parameters return ``(status, value)``.  ``GemmAmax`` is
a convenience holder of a plan and its workspace for torch tensors.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB, build  # noqa: F401

BSG_OK = 0
BSG_ERR_INVALID_ARG = 1
BSG_ERR_UNSUPPORTED = 2
BSG_ERR_ALIGNMENT = 3
BSG_ERR_ARCH = 4
BSG_ERR_WORKSPACE = 5
BSG_ERR_CUDA = 6
BSG_ERR_DEVICE_TIMEOUT = 7

BSG_E4M3 = 0
BSG_E5M2 = 1
BSG_E2M1 = 2
BSG_UE8M0 = 3
BSG_F32 = 4
BSG_F16 = 5
BSG_BF16 = 6

DTYPE = {"e4m3": BSG_E4M3, "e5m2": BSG_E5M2, "e2m1": BSG_E2M1, "ue8m0": BSG_UE8M0,
         "f32": BSG_F32, "f16": BSG_F16, "bf16": BSG_BF16}


class bsg_problem(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("L", ctypes.c_int64), ("a_dtype", ctypes.c_int32), ("b_dtype", ctypes.c_int32),
                ("sf_dtype", ctypes.c_int32), ("c_dtype", ctypes.c_int32),
                ("a_major", ctypes.c_char), ("b_major", ctypes.c_char),
                ("c_major", ctypes.c_char), ("reserved0", ctypes.c_char),
                ("sf_vec_size", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("cluster_m", ctypes.c_int32),
                ("cluster_n", ctypes.c_int32)]


class bsg_plan_info(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("tile_k_bytes", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
                ("mma_kind", ctypes.c_int32), ("cluster_m", ctypes.c_int32),
                ("kernel_name", ctypes.c_char * 64), ("half_tiles", ctypes.c_int32),
                ("k_split_tiles", ctypes.c_int32)]


BSG_QUANT_ROWWISE = 0
BSG_QUANT_COLWISE = 1
DIRECTION = {"row": BSG_QUANT_ROWWISE, "col": BSG_QUANT_COLWISE}


class bsg_quant_problem(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("L", ctypes.c_int64),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("sf_vec_size", ctypes.c_int), ("direction", ctypes.c_int)]


class bsg_device_buffers(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("SFA", ctypes.c_void_p),
                ("SFB", ctypes.c_void_p), ("C", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t)]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(
            "libbsgemm.so is missing: build the CUDA library first "
            "(block_scaled_precision_04_gb300.build()); there is no fallback path")
    lib = ctypes.CDLL(LIB)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.bsg_status_string.argtypes = [i32]
    lib.bsg_status_string.restype = ctypes.c_char_p
    lib.bsg_problem_check.argtypes = [ctypes.POINTER(bsg_problem)]
    lib.bsg_plan_create.argtypes = [ctypes.POINTER(bsg_problem), i32, ctypes.POINTER(vp)]
    lib.bsg_plan_workspace_size.argtypes = [vp, ctypes.POINTER(sz)]
    lib.bsg_workspace_init.argtypes = [vp, vp, sz, vp]
    lib.bsg_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.bsg_run_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(bsg_device_buffers),
                                 vp]
    lib.bsg_check_device_status.argtypes = [vp, vp, vp]
    lib.bsg_run_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.bsg_plan_describe.argtypes = [vp, ctypes.POINTER(bsg_plan_info)]
    lib.bsg_plan_destroy.argtypes = [vp]
    lib.bsg_plan_destroy.restype = None
    qp = ctypes.POINTER(bsg_quant_problem)
    lib.bsg_quant_check.argtypes = [qp]
    lib.bsg_quant_sizes.argtypes = [qp, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.bsg_quantize.argtypes = [qp, vp, vp, vp, vp]
    for name in ("bsg_problem_check", "bsg_plan_create", "bsg_plan_workspace_size",
                 "bsg_workspace_init", "bsg_run", "bsg_run_host", "bsg_check_device_status",
                 "bsg_run_noalloc",
                 "bsg_plan_describe", "bsg_quant_check", "bsg_quant_sizes", "bsg_quantize"):
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def make_problem(M, N, K, L, a_dtype="e4m3", b_dtype="e4m3", sf_vec_size=32, c_dtype="f32",
                 c_major="n", sf_dtype="ue8m0", a_major="k", b_major="k", tile_m=0, tile_n=0,
                 cluster_m=0, cluster_n=0) -> bsg_problem:
    """A bsg_problem from Python values (dtype names as in DTYPE, or the enum ints)."""
    d = lambda x: DTYPE[x] if isinstance(x, str) else int(x)
    return bsg_problem(int(M), int(N), int(K), int(L), d(a_dtype), d(b_dtype), d(sf_dtype),
                       d(c_dtype), a_major.encode(), b_major.encode(), c_major.encode(), b"\0",
                       int(sf_vec_size), int(tile_m), int(tile_n), int(cluster_m), int(cluster_n))


def problem_bytes(problem: bsg_problem) -> dict:
    """Bytes each tensor of `problem` spans in the library's layouts: A, B
    (codes; packed E2M1 two per byte), SFA, SFB (whole 128-row x 4-block
    scale atoms of 512 bytes) and C."""
    cdiv = lambda a, b: -(-a // b)
    fp4 = problem.a_dtype == BSG_E2M1
    kb = problem.K // 2 if fp4 else problem.K
    t_k = cdiv(problem.K, 4 * problem.sf_vec_size)
    item = {BSG_F32: 4, BSG_F16: 2, BSG_BF16: 2}.get(problem.c_dtype, 1)
    c = problem.L * problem.M * problem.N * item
    if problem.c_dtype == BSG_E2M1:
        c //= 2
    return {"A": problem.L * problem.M * kb, "B": problem.L * problem.N * kb,
            "SFA": problem.L * cdiv(problem.M, 128) * t_k * 512,
            "SFB": problem.L * cdiv(problem.N, 128) * t_k * 512, "C": c}


def bsg_status_string(status: int) -> str:
    return library().bsg_status_string(int(status)).decode()


def bsg_problem_check(problem: bsg_problem) -> int:
    return library().bsg_problem_check(ctypes.byref(problem))


def bsg_plan_create(problem: bsg_problem, device: int = 0):
    plan = ctypes.c_void_p()
    st = library().bsg_plan_create(ctypes.byref(problem), int(device), ctypes.byref(plan))
    return st, plan


def bsg_plan_workspace_size(plan):
    n = ctypes.c_size_t()
    st = library().bsg_plan_workspace_size(plan, ctypes.byref(n))
    return st, n.value


def bsg_workspace_init(plan, workspace: int, ws_bytes: int, stream: int = 0) -> int:
    return library().bsg_workspace_init(plan, ctypes.c_void_p(workspace), ws_bytes,
                                        ctypes.c_void_p(stream))


def bsg_run(plan, A: int, B: int, SFA: int, SFB: int, C: int, amax: int, workspace: int,
            ws_bytes: int, stream: int = 0) -> int:
    v = ctypes.c_void_p
    return library().bsg_run(plan, v(A), v(B), v(SFA), v(SFB), v(C), v(amax), v(workspace),
                             ws_bytes, v(stream))


def bsg_run_host(plan, hA: int, hB: int, hSFA: int, hSFB: int, hC: int, h_amax: int,
                 dev: bsg_device_buffers, stream: int = 0) -> int:
    v = ctypes.c_void_p
    return library().bsg_run_host(plan, v(hA), v(hB), v(hSFA), v(hSFB), v(hC), v(h_amax),
                                  ctypes.byref(dev), v(stream))


def bsg_run_noalloc(plan, A: int, B: int, SFA: int, SFB: int, C: int, amax: int,
                    stream: int = 0) -> int:
    """bsg_run for callers that cannot allocate: the workspace is a fixed
    array inside the library (see include/bsgemm.h)."""
    v = ctypes.c_void_p
    return library().bsg_run_noalloc(plan, v(A), v(B), v(SFA), v(SFB), v(C), v(amax), v(stream))


def bsg_check_device_status(plan, workspace: int, stream: int = 0) -> int:
    return library().bsg_check_device_status(plan, ctypes.c_void_p(workspace),
                                             ctypes.c_void_p(stream))


def bsg_plan_describe(plan):
    info = bsg_plan_info()
    st = library().bsg_plan_describe(plan, ctypes.byref(info))
    out = {f: getattr(info, f) for f, _ in bsg_plan_info._fields_}
    out["kernel_name"] = info.kernel_name.decode()
    return st, out


def bsg_plan_destroy(plan) -> None:
    library().bsg_plan_destroy(plan)


class BsgError(RuntimeError):
    def __init__(self, where: str, status: int):
        super().__init__(f"{where}: {bsg_status_string(status)} (status {status})")
        self.status = status


def check(status: int, where: str = "bsgemm") -> None:
    if status != BSG_OK:
        raise BsgError(where, status)


class GemmAmax:
    """A plan plus its workspace, run on torch CUDA tensors.

    ``run(A, B, SFA, SFB, C, amax)`` takes contiguous uint8 tensors for the
    codes and the physical scale atoms, C of the plan's dtype and layout and a
    one-element fp32 amax, all on the plan's device, and enqueues one launch
    on torch's current stream."""

    def __init__(self, problem: bsg_problem, device: int = 0):
        import torch
        self.problem = problem
        self.device = int(device)
        st, self.plan = bsg_plan_create(problem, self.device)
        check(st, "bsg_plan_create")
        st, self.ws_bytes = bsg_plan_workspace_size(self.plan)
        check(st, "bsg_plan_workspace_size")
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8,
                                     device=f"cuda:{self.device}")
        check(bsg_workspace_init(self.plan, self.workspace.data_ptr(), self.ws_bytes,
                                 torch.cuda.current_stream(self.device).cuda_stream),
              "bsg_workspace_init")

    def describe(self) -> dict:
        st, info = bsg_plan_describe(self.plan)
        check(st, "bsg_plan_describe")
        return info

    def run(self, A, B, SFA, SFB, C, amax, stream=None) -> None:
        import torch
        need = problem_bytes(self.problem)
        need["amax"] = 4
        for name, t in (("A", A), ("B", B), ("SFA", SFA), ("SFB", SFB), ("C", C), ("amax", amax)):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CUDA tensor")
            if t.numel() * t.element_size() < need[name]:
                raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, "
                                 f"the problem needs {need[name]}")
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        check(bsg_run(self.plan, A.data_ptr(), B.data_ptr(), SFA.data_ptr(), SFB.data_ptr(),
                      C.data_ptr(), amax.data_ptr(), self.workspace.data_ptr(), self.ws_bytes, s),
              "bsg_run")

    def device_status(self, stream=None) -> int:
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        return bsg_check_device_status(self.plan, self.workspace.data_ptr(), s)

    def close(self) -> None:
        if getattr(self, "plan", None):
            bsg_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------- quantizer

def make_quant_problem(rows, cols, L=1, in_dtype="f32", out_dtype="e4m3",
                       sf_vec_size=32, direction="row") -> bsg_quant_problem:
    """A bsg_quant_problem; ``direction`` is "row" (blocks along each row) or
    "col" (blocks of 32 down each column), or the enum value."""
    d = lambda x: DTYPE[x] if isinstance(x, str) else int(x)
    dr = DIRECTION[direction] if isinstance(direction, str) else int(direction)
    return bsg_quant_problem(int(rows), int(cols), int(L), d(in_dtype), d(out_dtype),
                             int(sf_vec_size), dr)


def bsg_quant_check(q: bsg_quant_problem) -> int:
    return library().bsg_quant_check(ctypes.byref(q))


def bsg_quant_sizes(q: bsg_quant_problem):
    cb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = library().bsg_quant_sizes(ctypes.byref(q), ctypes.byref(cb), ctypes.byref(sb))
    return st, (cb.value, sb.value)


def bsg_quantize(q: bsg_quant_problem, X: int, codes: int, sf: int, stream: int = 0) -> int:
    return library().bsg_quantize(ctypes.byref(q), X, codes, sf, stream)


def quantize(X, out_dtype="e4m3", sf_vec_size=32, codes=None, sf=None, stream=None,
             direction="row"):
    """Quantize a contiguous CUDA tensor X (L, rows, cols) or (rows, cols) of
    float32 or bfloat16 into (codes, sf) uint8 tensors (allocated when not
    given); one launch on torch's current stream.  ``direction="col"`` puts
    the blocks down the columns: the codes are then the GEMM's MN-major
    operand (rows = K) and sf its scale atoms."""
    import torch
    if not X.is_cuda or not X.is_contiguous():
        raise ValueError("X must be a contiguous CUDA tensor")
    shape = tuple(X.shape) if X.dim() == 3 else (1,) + tuple(X.shape)
    in_dtype = {torch.float32: "f32", torch.bfloat16: "bf16"}.get(X.dtype)
    if in_dtype is None:
        raise ValueError("X must be float32 or bfloat16")
    q = make_quant_problem(shape[1], shape[2], shape[0], in_dtype, out_dtype, sf_vec_size,
                           direction)
    st, (cb, sb) = bsg_quant_sizes(q)
    check(st, "bsg_quant_sizes")
    if codes is None:
        codes = torch.empty(cb, dtype=torch.uint8, device=X.device)
    if sf is None:
        sf = torch.empty(sb, dtype=torch.uint8, device=X.device)
    if codes.numel() < cb or sf.numel() < sb:
        raise ValueError("codes / sf buffers too small")
    s = stream if stream is not None else torch.cuda.current_stream(X.device).cuda_stream
    check(bsg_quantize(q, X.data_ptr(), codes.data_ptr(), sf.data_ptr(), s), "bsg_quantize")
    return codes, sf

