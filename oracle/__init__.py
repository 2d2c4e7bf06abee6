"""CPU oracle for the block-scaled GEMM + Amax ("GEMM + Amax (SM100)").

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (the CUDA library under ``block_scaled_precision_04_gb300``) never
imports it, and this package imports nothing from there.

The arithmetic lives in ``bsg_oracle.c`` (plain C, IEEE double); this module
builds it with gcc, loads it with ctypes and marshals numpy arrays.  The
functions follow the page's section "Equations":

* ``dequantize``    -- Ahat = dec(A) * 2^(SFA - 127) per sf_vec_size K-block
* ``gemm``          -- C = sum_k Ahat * Bhat (double), and S = sum_k |Ahat * Bhat|
* ``gemm_sample``   -- the same sums at chosen (m, n, l) points
* ``round_to``      -- C rounded to the output dtype (round-to-nearest-even)
* ``ulp``, ``tolerance`` -- tau = 1e-5 * S + ulp_c(|C_ref|)
* ``reference``     -- C_ref, S, tau and Amax = max |C_ref| for a whole problem
* ``quantize``      -- the row upstream of the GEMM: real values -> element
  codes + E8M0 scales in the atom layout ("GEMM + RoPE + MXFP8 Projection
  (SM100)", "Equations"; the block-scale rule is the reading stated in
  bsg_oracle.c); ``quantize_value`` rounds one scaled value
* ``quantize_colwise`` -- the same rule with blocks down the rows (the
  page's S-direction), codes in X's layout = the GEMM's MN-major operand,
  scales in the atom layout keyed by column

Parity unpinned: the split of a row index mn = m0 + 32*m1 inside a 128-row
scale atom is the column-major reading of the atom's shape (32, 4); the pages
give the shape and the permutation, not this split.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsg_oracle.c")
_LIB = os.path.join(_HERE, "libbsgoracle.so")

DTYPES = {"e4m3": 0, "e5m2": 1, "e2m1": 2, "ue8m0": 3, "f32": 4, "f16": 5, "bf16": 6}
REL_TOL = 1e-5

_lib = None


def build(force: bool = False) -> str:
    """Compile bsg_oracle.c into libbsgoracle.so next to it (gcc, -O2, no
    floating-point contraction or reassociation)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64p = ctypes.POINTER(ctypes.c_int64)
    u8p = ctypes.c_void_p
    dp = ctypes.c_void_p
    lib.bsgo_decode_table.argtypes = [ctypes.c_int, dp]
    lib.bsgo_decode_table.restype = ctypes.c_int
    lib.bsgo_sf_offset.argtypes = [ctypes.c_int64] * 5
    lib.bsgo_sf_offset.restype = ctypes.c_int64
    lib.bsgo_dequantize.argtypes = [u8p, ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, dp]
    lib.bsgo_dequantize.restype = ctypes.c_int
    lib.bsgo_num_threads.argtypes = [ctypes.c_int]
    lib.bsgo_num_threads.restype = ctypes.c_int
    lib.bsgo_gemm.argtypes = [i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              u8p, u8p, u8p, u8p, dp, dp, ctypes.c_int]
    lib.bsgo_gemm.restype = ctypes.c_int
    lib.bsgo_gemm_rows.argtypes = [i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   u8p, u8p, u8p, u8p, ctypes.c_int64, ctypes.c_int64,
                                   dp, dp, ctypes.c_int]
    lib.bsgo_gemm_rows.restype = ctypes.c_int
    lib.bsgo_gemm_sample.argtypes = [i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, u8p, u8p, u8p, u8p, i64p, ctypes.c_int64,
                                     dp, dp, ctypes.c_int]
    lib.bsgo_gemm_sample.restype = ctypes.c_int
    lib.bsgo_round.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.bsgo_round.restype = ctypes.c_double
    lib.bsgo_ulp.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.bsgo_ulp.restype = ctypes.c_double
    lib.bsgo_round_array.argtypes = [dp, ctypes.c_int64, ctypes.c_int, dp]
    lib.bsgo_round_array.restype = ctypes.c_int
    lib.bsgo_tolerance.argtypes = [dp, dp, ctypes.c_int64, ctypes.c_int, ctypes.c_double, dp]
    lib.bsgo_tolerance.restype = ctypes.c_int
    lib.bsgo_quantize_value.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.bsgo_quantize_value.restype = ctypes.c_int
    lib.bsgo_quantize.argtypes = [dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_int, ctypes.c_int, u8p, u8p]
    lib.bsgo_quantize.restype = ctypes.c_int
    lib.bsgo_quantize_colwise.argtypes = [dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_int, u8p, u8p]
    lib.bsgo_quantize_colwise.restype = ctypes.c_int
    _lib = lib
    return lib


def _u8(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("codes and scales are passed as uint8 bytes, got %s" % a.dtype)
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _mn(major: str, mn_name: str) -> int:
    """1 for an operand stored with its M (N) rows contiguous, 0 for k-major."""
    if major == "k":
        return 0
    if major == mn_name:
        return 1
    raise ValueError("operand major must be 'k' or %r, got %r" % (mn_name, major))


def _dims(M, N, K, L, a_major="k", b_major="k"):
    return (ctypes.c_int64 * 6)(int(M), int(N), int(K), int(L), _mn(a_major, "m"),
                                _mn(b_major, "n"))


def num_threads(requested: int = 0) -> int:
    """Threads the oracle uses for `requested` (0 = every core it may run on)."""
    return _load().bsgo_num_threads(int(requested))


def decode_table(dtype: str) -> np.ndarray:
    """Value of every code of `dtype` (256 entries, 16 for e2m1); NaN codes give NaN."""
    out = np.empty(256, dtype=np.float64)
    n = _load().bsgo_decode_table(DTYPES[dtype], _ptr(out))
    if n < 0:
        raise ValueError(dtype)
    return out[:n].copy()


def sf_offset(mn: int, kb: int, l: int, t_mn: int, t_k: int) -> int:
    """Byte offset of scale (mn, kb, l) in the physical (L, t_mn, t_k, 32, 4, 4) tensor."""
    return int(_load().bsgo_sf_offset(mn, kb, l, t_mn, t_k))


def dequantize(codes: np.ndarray, dtype: str, sf: np.ndarray, sfv: int, rows: int, K: int,
               L: int, sf_dtype: str = "ue8m0") -> np.ndarray:
    """Dequantized operand, shape (L, rows, K), float64."""
    codes, sf = _u8(codes), _u8(sf)
    out = np.empty((L, rows, K), dtype=np.float64)
    rc = _load().bsgo_dequantize(_ptr(codes), DTYPES[dtype], _ptr(sf), DTYPES[sf_dtype],
                                 int(sfv), int(rows), int(K), int(L), _ptr(out))
    if rc != 0:
        raise ValueError("bad dequantize arguments")
    return out


def gemm(M, N, K, L, a_dtype, b_dtype, sfv, A, B, SFA, SFB, sf_dtype="ue8m0",
         rows=None, nthreads=0, want_s=True, a_major="k", b_major="k"):
    """C[l, m, n] = sum_k Ahat[m,k,l] Bhat[n,k,l] in double, and S = sum_k |Ahat Bhat|.

    A is k-major bytes (L, M, K) (K/2 for E2M1) or, with ``a_major="m"``
    (FP8 only), m-major bytes (L, K, M); B likewise with ``b_major="n"``.
    ``rows=(m0, m1)`` restricts to rows m0 <= m < m1 (every batch).
    Returns (C, S, threads_used); S is None when ``want_s`` is false."""
    A, B, SFA, SFB = _u8(A), _u8(B), _u8(SFA), _u8(SFB)
    m0, m1 = (0, M) if rows is None else rows
    C = np.empty((L, m1 - m0, N), dtype=np.float64)
    S = np.empty_like(C) if want_s else None
    nt = _load().bsgo_gemm_rows(_dims(M, N, K, L, a_major, b_major), DTYPES[a_dtype],
                                DTYPES[b_dtype],
                                DTYPES[sf_dtype], int(sfv), _ptr(A), _ptr(B), _ptr(SFA),
                                _ptr(SFB), int(m0), int(m1), _ptr(C),
                                _ptr(S) if S is not None else None, int(nthreads))
    if nt < 0:
        raise ValueError("bad gemm arguments")
    return C, S, nt


def gemm_sample(M, N, K, L, a_dtype, b_dtype, sfv, A, B, SFA, SFB, mnl, sf_dtype="ue8m0",
                nthreads=0, a_major="k", b_major="k"):
    """The sums at points mnl (an (n, 3) int array of (m, n, l)).  Returns (C, S)."""
    A, B, SFA, SFB = _u8(A), _u8(B), _u8(SFA), _u8(SFB)
    mnl = np.ascontiguousarray(mnl, dtype=np.int64).reshape(-1, 3)
    C = np.empty(len(mnl), dtype=np.float64)
    S = np.empty(len(mnl), dtype=np.float64)
    nt = _load().bsgo_gemm_sample(_dims(M, N, K, L, a_major, b_major), DTYPES[a_dtype],
                                  DTYPES[b_dtype],
                                  DTYPES[sf_dtype], int(sfv), _ptr(A), _ptr(B), _ptr(SFA),
                                  _ptr(SFB), mnl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                  len(mnl), _ptr(C), _ptr(S), int(nthreads))
    if nt < 0:
        raise ValueError("bad sample arguments")
    return C, S


def round_to(x: np.ndarray, c_dtype: str) -> np.ndarray:
    """x (float64) rounded to c_dtype, round-to-nearest-even, returned as float64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    if _load().bsgo_round_array(_ptr(x), x.size, DTYPES[c_dtype], _ptr(out)) != 0:
        raise ValueError(c_dtype)
    return out


def ulp(x, c_dtype: str):
    """Spacing of c_dtype at |x|."""
    lib = _load()
    if np.isscalar(x):
        return lib.bsgo_ulp(float(x), DTYPES[c_dtype])
    return np.vectorize(lambda v: lib.bsgo_ulp(float(v), DTYPES[c_dtype]))(x)


def tolerance(cref: np.ndarray, S: np.ndarray, c_dtype: str, rel: float = REL_TOL):
    """tau = rel * S + ulp_c(|cref|), elementwise."""
    cref = np.ascontiguousarray(cref, dtype=np.float64)
    S = np.ascontiguousarray(S, dtype=np.float64)
    tau = np.empty_like(cref)
    if _load().bsgo_tolerance(_ptr(cref), _ptr(S), cref.size, DTYPES[c_dtype], float(rel),
                              _ptr(tau)) != 0:
        raise ValueError(c_dtype)
    return tau


def reference(M, N, K, L, a_dtype, b_dtype, sfv, A, B, SFA, SFB, c_dtype, sf_dtype="ue8m0",
              nthreads=0, a_major="k", b_major="k"):
    """Everything a parity check needs for a whole problem, arrays shaped (L, M, N):
    ``c`` (C_ref rounded to c_dtype), ``exact`` (the double sum), ``s``, ``tau`` and
    ``amax`` (max |C_ref|)."""
    C, S, _ = gemm(M, N, K, L, a_dtype, b_dtype, sfv, A, B, SFA, SFB, sf_dtype=sf_dtype,
                   nthreads=nthreads, a_major=a_major, b_major=b_major)
    cref = round_to(C, c_dtype)
    tau = tolerance(cref, S, c_dtype)
    return {"c": cref, "exact": C, "s": S, "tau": tau, "amax": float(np.max(np.abs(cref)))}


def quant_sizes(rows: int, cols: int, L: int, out_dtype: str, sfv: int):
    """(code bytes, scale bytes) of a quantized (rows, cols, L) tensor; the
    scales cover whole (padded) atoms."""
    t_r = -(-rows // 128)
    t_k = -(-(cols // sfv) // 4)
    code_bytes = L * rows * (cols // 2 if out_dtype == "e2m1" else cols)
    return code_bytes, L * t_r * t_k * 512


def quantize_value(y: float, out_dtype: str) -> int:
    """Code of the out_dtype value nearest to y (ties to even, saturating)."""
    c = _load().bsgo_quantize_value(float(y), DTYPES[out_dtype])
    if c < 0:
        raise ValueError(out_dtype)
    return int(c)


def quantize(X: np.ndarray, out_dtype: str, sfv: int):
    """X (L, rows, cols) real values -> (codes uint8 (L, rows, cols or cols/2),
    scales uint8 (L, t_r, t_k, 32, 4, 4))."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    if X.ndim == 2:
        X = X[None]
    L, rows, cols = X.shape
    code_bytes, sf_bytes = quant_sizes(rows, cols, L, out_dtype, sfv)
    codes = np.zeros(code_bytes, dtype=np.uint8)
    sf = np.zeros(sf_bytes, dtype=np.uint8)
    rc = _load().bsgo_quantize(_ptr(X), int(rows), int(cols), int(L), DTYPES[out_dtype],
                               int(sfv), _ptr(codes), _ptr(sf))
    if rc != 0:
        raise ValueError("unsupported quantize request")
    t_r = -(-rows // 128)
    t_k = -(-(cols // sfv) // 4)
    return (codes.reshape(L, rows, -1), sf.reshape(L, t_r, t_k, 32, 4, 4))



def quant_colwise_sizes(rows: int, cols: int, L: int) -> tuple[int, int]:
    """Bytes of the columnwise codes and of its padded scale atom tensor
    (blocks of 32 rows; scale atoms over ceil(cols/128) x ceil(rows/128))."""
    return L * rows * cols, L * (-(-cols // 128)) * (-(-(rows // 32) // 4)) * 512


def quantize_colwise(X: np.ndarray, out_dtype: str, sfv: int = 32):
    """X (L, rows, cols) real values, blocks of sfv rows down each column ->
    (codes uint8 (L, rows, cols), scales uint8 (L, t_c, t_k, 32, 4, 4)) with
    t_c = ceil(cols/128), t_k = ceil(rows/sfv/4).  Read as a GEMM operand the
    codes are MN-major (rows = K, cols = M or N)."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    if X.ndim == 2:
        X = X[None]
    L, rows, cols = X.shape
    code_bytes, sf_bytes = quant_colwise_sizes(rows, cols, L)
    codes = np.zeros(code_bytes, dtype=np.uint8)
    sf = np.zeros(sf_bytes, dtype=np.uint8)
    rc = _load().bsgo_quantize_colwise(_ptr(X), int(rows), int(cols), int(L),
                                       DTYPES[out_dtype], int(sfv), _ptr(codes), _ptr(sf))
    if rc != 0:
        raise ValueError("unsupported columnwise quantize request")
    t_c = -(-cols // 128)
    t_k = -(-(rows // sfv) // 4)
    return codes.reshape(L, rows, cols), sf.reshape(L, t_c, t_k, 32, 4, 4)
