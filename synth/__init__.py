"""Seeded synthetic inputs for the block-scaled GEMM + Amax.

This module only draws random numbers and encodes them into the input
formats the operation consumes (FP8/FP4 codes plus E8M0 or E4M3 block scales
laid out in the 128-row scale atoms).  It holds none of the operation's own
arithmetic: no decoding tables, no dot products, no reductions (torch's
float8 casts encode, and for the E4M3 scale recipe decode, single values).  Both the CUDA path's tests and
the CPU oracle are fed from here; neither of them is imported.

Layouts produced (page "GEMM + Amax (SM100)", section "Parameters"):

* ``A``: uint8, shape (L, M, K) -- k-major (M, K, L) with strides (K, 1, M*K);
  (L, M, K/2) for packed E2M1, element 2i in the low nibble.
* ``B``: uint8, shape (L, N, K) or (L, N, K/2), likewise.
* ``SFA`` / ``SFB``: uint8, the C-contiguous physical scale tensor
  (L, ceil(MN/128), ceil(K/(4*sfv)), 32, 4, 4), whose permutation by
  (3, 4, 1, 5, 2, 0) is the logical (32, 4, ceil(MN/128), 4, ceil(K/(4*sfv)), L)
  view ("Using JAX arrays").  Padding entries (rows past MN, K-blocks past
  ceil(K/sfv)) hold 127 (a scale of 1).

Workloads (seed = 1000 + workload number):

1. E4M3 256x256x256, L=1: codes uniform over the 254 finite E4M3 bytes,
   scale bytes uniform in [124, 130]; C fp32 n-major.
2. MXFP8 4096^3, L=1: A, B ~ N(0,1), per-32 K-block E4M3 with scale
   2^(floor(log2(block amax)) - 8); C bf16 n-major.
3. Batched MXFP8 L=8, 2048x2048x8192: A ~ N(0,1) with ceil(1% of M) rows
   per batch multiplied by 64 before quantising, A to E5M2, B to E4M3;
   C fp32 n-major.
4. FP4 E2M1 8192^3, L=1, sf_vec_size 16, scale 2^(floor(log2(block amax)) - 2);
   C bf16 n-major.
5. Ragged MXFP8 L=2, 8000x1000x7168: A ~ U[-1,1], B ~ N(0, 0.02), E4M3;
   C fp32 m-major.
6. NVFP4 8192^3, L=1: A, B ~ N(0,1), per-16 K-block E2M1 with an E4M3 scale
   byte = the block amax / 6 rounded to E4M3 (nearest, ties to even; at least
   the smallest subnormal, 1.0 for an all-zero block), each element divided
   by the decoded scale, saturated to +-6 and rounded to E2M1; C bf16 n-major.
7. MXFP8 4096^3 with MN-major operands: workload 2's recipe, A stored m-major
   (strides (1, M, M*K)) and B n-major.

The exponent offset of a block scale is the element format's largest
exponent (E4M3 8, E5M2 15, E2M1 2); the scaled block is saturated to the
format's largest finite value and rounded to nearest, ties to even.  A block
whose amax is zero gets the scale byte 127.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

ELEM_EMAX = {"e4m3": 8, "e5m2": 15, "e2m1": 2}
ELEM_MAX = {"e4m3": 448.0, "e5m2": 57344.0, "e2m1": 6.0}
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclasses.dataclass(frozen=True)
class Problem:
    M: int
    N: int
    K: int
    L: int
    a_dtype: str = "e4m3"
    b_dtype: str = "e4m3"
    sfv: int = 32
    c_dtype: str = "f32"
    c_major: str = "n"
    sf_dtype: str = "ue8m0"
    a_major: str = "k"   # "k": A bytes (L, M, K); "m" (FP8 only): (L, K, M)
    b_major: str = "k"   # "k": B bytes (L, N, K); "n" (FP8 only): (L, K, N)

    @property
    def t_m(self) -> int:
        return _cdiv(self.M, 128)

    @property
    def t_n(self) -> int:
        return _cdiv(self.N, 128)

    @property
    def t_k(self) -> int:
        return _cdiv(self.K, 4 * self.sfv)

    def row_bytes(self, dtype: str) -> int:
        return self.K // 2 if dtype == "e2m1" else self.K

    @property
    def c_itemsize(self) -> float:
        return {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1, "e5m2": 1, "e2m1": 0.5}[self.c_dtype]

    def describe(self) -> str:
        ab = self.a_dtype if self.a_dtype == self.b_dtype else f"{self.a_dtype}x{self.b_dtype}"
        return (f"{ab} M={self.M} N={self.N} K={self.K} L={self.L} sfv={self.sfv} "
                f"sf={self.sf_dtype} A {self.a_major}-major B {self.b_major}-major "
                f"C={self.c_dtype} {self.c_major}-major")


@dataclasses.dataclass
class Inputs:
    problem: Problem
    A: np.ndarray
    B: np.ndarray
    SFA: np.ndarray
    SFB: np.ndarray
    name: str = ""


WORKLOADS = {
    1: ("e4m3-256^3-uniform-codes",
        Problem(256, 256, 256, 1, "e4m3", "e4m3", 32, "f32", "n")),
    2: ("mxfp8-4096^3-bf16",
        Problem(4096, 4096, 4096, 1, "e4m3", "e4m3", 32, "bf16", "n")),
    3: ("mxfp8-batched-L8-2048x2048x8192-e5m2xe4m3-outliers",
        Problem(2048, 2048, 8192, 8, "e5m2", "e4m3", 32, "f32", "n")),
    4: ("mxfp4-8192^3-sfv16-bf16",
        Problem(8192, 8192, 8192, 1, "e2m1", "e2m1", 16, "bf16", "n")),
    5: ("mxfp8-ragged-L2-8000x1000x7168-mmajor",
        Problem(8000, 1000, 7168, 2, "e4m3", "e4m3", 32, "f32", "m")),
    6: ("nvfp4-8192^3-sfv16-e4m3-scales-bf16",
        Problem(8192, 8192, 8192, 1, "e2m1", "e2m1", 16, "bf16", "n", sf_dtype="e4m3")),
    7: ("mxfp8-4096^3-a-mmajor-b-nmajor-bf16",
        Problem(4096, 4096, 4096, 1, "e4m3", "e4m3", 32, "bf16", "n", a_major="m", b_major="n")),
}

E4M3_ONE = 0x38  # the E4M3 byte of 1.0, the padding scale of E4M3 atoms


# ---------------------------------------------------------------- encoding

def _encode_fp8(y: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values already inside the format's range -> FP8 bytes (RNE)."""
    tdt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(tdt).view(
        torch.uint8).numpy()


def _encode_e2m1(y: np.ndarray) -> np.ndarray:
    """float32 values in [-6, 6] -> 4-bit E2M1 codes (one per uint8), RNE."""
    a = np.abs(y).astype(np.float32)
    i = np.searchsorted(_E2M1_GRID, a, side="right") - 1
    i = np.clip(i, 0, 7)
    j = np.minimum(i + 1, 7)
    lo, hi = _E2M1_GRID[i], _E2M1_GRID[j]
    d_lo, d_hi = a - lo, hi - a
    up = (j != i) & ((d_hi < d_lo) | ((d_hi == d_lo) & (j % 2 == 0)))
    code = np.where(up, j, i).astype(np.uint8)
    code |= np.where(y < 0, np.uint8(8), np.uint8(0)).astype(np.uint8)
    return code


def _pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """(..., K) 4-bit codes -> (..., K/2) bytes, element 2i in the low nibble."""
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return (lo | (hi << 4)).astype(np.uint8)


def quantize_blocks(x: np.ndarray, dtype: str, sfv: int):
    """x: (R, K) float32 with K % sfv == 0.  Returns (codes (R, K or K/2) uint8,
    scale bytes (R, K/sfv) uint8)."""
    R, K = x.shape
    xb = x.reshape(R, K // sfv, sfv)
    amax = np.max(np.abs(xb), axis=2)
    _, e = np.frexp(amax)  # amax = f * 2^e, f in [0.5, 1) => floor(log2 amax) = e - 1
    sf = (e.astype(np.int64) - 1) - ELEM_EMAX[dtype] + 127
    sf = np.where(amax > 0, sf, 127)
    sf = np.clip(sf, 1, 254).astype(np.uint8)
    inv = np.ldexp(np.float32(1.0), (127 - sf.astype(np.int32))).astype(np.float32)
    y = xb * inv[:, :, None]
    m = ELEM_MAX[dtype]
    y = np.clip(y, -m, m).reshape(R, K)
    if dtype == "e2m1":
        codes = _pack_e2m1(_encode_e2m1(y))
    else:
        codes = _encode_fp8(y, dtype)
    return codes, sf


def quantize_blocks_e4m3_scale(x: np.ndarray, sfv: int = 16):
    """NVFP4-style: x (R, K) float32, K % sfv == 0 -> (packed E2M1 codes
    (R, K/2), E4M3 scale bytes (R, K/sfv)) by the workload-6 recipe."""
    R, K = x.shape
    xb = x.reshape(R, K // sfv, sfv)
    amax = np.max(np.abs(xb), axis=2)
    sb = _encode_fp8(np.minimum(amax / np.float32(6.0), np.float32(448.0)), "e4m3")
    sb = np.where(sb == 0, np.uint8(1), sb)
    sb = np.where(amax > 0, sb, np.uint8(E4M3_ONE)).astype(np.uint8)
    dec = torch.from_numpy(sb).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    y = np.clip(xb / dec[:, :, None], -6.0, 6.0).reshape(R, K)
    return _pack_e2m1(_encode_e2m1(y)), sb


def pack_scale_atoms(sf: np.ndarray, rows: int, K: int, sfv: int, pad: int = 127) -> np.ndarray:
    """Logical scales (L, rows, ceil(K/sfv)) -> physical (L, T, T_k, 32, 4, 4) bytes.

    Row r = 128*t + 32*m1 + m0 goes to [l, t, kt, m0, m1, kin] for K-block
    kb = 4*kt + kin."""
    L = sf.shape[0]
    t, t_k = _cdiv(rows, 128), _cdiv(K, 4 * sfv)
    full = np.full((L, t * 128, t_k * 4), pad, dtype=np.uint8)
    full[:, :rows, :sf.shape[2]] = sf
    x = full.reshape(L, t, 4, 32, t_k, 4)          # [l, t, m1, m0, kt, kin]
    x = x.transpose(0, 1, 4, 3, 2, 5)               # [l, t, kt, m0, m1, kin]
    return np.ascontiguousarray(x)


def scale_shape(rows: int, K: int, sfv: int, L: int):
    return (L, _cdiv(rows, 128), _cdiv(K, 4 * sfv), 32, 4, 4)


# ---------------------------------------------------------------- workloads

_FINITE_E4M3 = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], dtype=np.uint8)


def to_major(codes: np.ndarray, major: str) -> np.ndarray:
    """k-major operand bytes (L, rows, K) in the stored layout: unchanged for
    "k", (L, K, rows) with the rows contiguous for "m" / "n" ("Parameters":
    strides (1, M, M*K))."""
    if major == "k":
        return codes
    return np.ascontiguousarray(codes.transpose(0, 2, 1))


def uniform_codes(p: Problem, seed: int, sf_lo: int = 124, sf_hi: int = 130) -> Inputs:
    """Codes uniform over the finite codes of each format; every scale byte
    (padding included) uniform in [sf_lo, sf_hi]."""
    rng = np.random.default_rng(seed)

    def codes(rows, dtype):
        if dtype == "e4m3":
            return _FINITE_E4M3[rng.integers(0, len(_FINITE_E4M3), size=(p.L, rows, p.K))]
        if dtype == "e5m2":
            fin = np.array([b for b in range(256) if (b & 0x7C) != 0x7C], dtype=np.uint8)
            return fin[rng.integers(0, len(fin), size=(p.L, rows, p.K))]
        c = rng.integers(0, 16, size=(p.L, rows, p.K)).astype(np.uint8)
        return _pack_e2m1(c)

    A = codes(p.M, p.a_dtype)
    B = codes(p.N, p.b_dtype)
    SFA = rng.integers(sf_lo, sf_hi + 1, size=scale_shape(p.M, p.K, p.sfv, p.L)).astype(np.uint8)
    SFB = rng.integers(sf_lo, sf_hi + 1, size=scale_shape(p.N, p.K, p.sfv, p.L)).astype(np.uint8)
    return Inputs(p, to_major(A, p.a_major), to_major(B, p.b_major), SFA, SFB)


def quantized(p: Problem, seed: int, a_dist: str = "normal", b_dist: str = "normal",
              b_sigma: float = 1.0, outlier_frac: float = 0.0, outlier_scale: float = 64.0
              ) -> Inputs:
    """Real-valued draws quantised per sf_vec_size K-block (see module doc)."""
    if p.K % p.sfv:
        raise ValueError("quantised workloads need K % sf_vec_size == 0")
    if p.sf_dtype == "e4m3":
        if p.a_dtype != "e2m1" or p.b_dtype != "e2m1":
            raise ValueError("E4M3 scales are for E2M1 operands")
        enc = lambda x, dtype: quantize_blocks_e4m3_scale(x, p.sfv)
    else:
        enc = lambda x, dtype: quantize_blocks(x, dtype, p.sfv)
    rng = np.random.default_rng(seed)
    a_bytes = p.row_bytes(p.a_dtype)
    b_bytes = p.row_bytes(p.b_dtype)
    A = np.empty((p.L, p.M, a_bytes), dtype=np.uint8)
    B = np.empty((p.L, p.N, b_bytes), dtype=np.uint8)
    sfa = np.empty((p.L, p.M, p.K // p.sfv), dtype=np.uint8)
    sfb = np.empty((p.L, p.N, p.K // p.sfv), dtype=np.uint8)
    for l in range(p.L):
        if a_dist == "uniform":
            x = rng.uniform(-1.0, 1.0, size=(p.M, p.K)).astype(np.float32)
        else:
            x = rng.standard_normal((p.M, p.K), dtype=np.float32)
        if outlier_frac > 0:
            n_out = int(math.ceil(outlier_frac * p.M))
            rows = rng.choice(p.M, size=n_out, replace=False)
            x[rows] *= np.float32(outlier_scale)
        A[l], sfa[l] = enc(x, p.a_dtype)
    for l in range(p.L):
        x = rng.standard_normal((p.N, p.K), dtype=np.float32)
        if b_sigma != 1.0:
            x *= np.float32(b_sigma)
        B[l], sfb[l] = enc(x, p.b_dtype)
    pad = E4M3_ONE if p.sf_dtype == "e4m3" else 127
    SFA = pack_scale_atoms(sfa, p.M, p.K, p.sfv, pad)
    SFB = pack_scale_atoms(sfb, p.N, p.K, p.sfv, pad)
    return Inputs(p, to_major(A, p.a_major), to_major(B, p.b_major), SFA, SFB)


def workload(number: int, seed: int | None = None, **shape) -> Inputs:
    """Inputs of workload `number` (1..7).  Keyword overrides (M, N, K, L)
    keep the recipe and change the shape (parity cases at reduced size);
    `seed` replaces the workload's own seed 1000 + number (the batches of
    another rank of a sharded run)."""
    name, p = WORKLOADS[number]
    if shape:
        p = dataclasses.replace(p, **shape)
    if seed is None:
        seed = 1000 + number
    if number == 1:
        inp = uniform_codes(p, seed)
    elif number == 2:
        inp = quantized(p, seed)
    elif number == 3:
        inp = quantized(p, seed, outlier_frac=0.01, outlier_scale=64.0)
    elif number == 4:
        inp = quantized(p, seed)
    elif number == 5:
        inp = quantized(p, seed, a_dist="uniform", b_sigma=0.02)
    elif number in (6, 7):
        inp = quantized(p, seed)
    else:
        raise KeyError(number)
    inp.name = name if not shape else name + "@" + ",".join(f"{k}={v}" for k, v in shape.items())
    return inp


def c_shape(p: Problem):
    """Memory shape of C: (L, M, N) for n-major, (L, N, M) for m-major; packed
    E2M1 C (n-major only) is (L, M, N/2) bytes."""
    if p.c_dtype == "e2m1":
        return (p.L, p.M, p.N // 2)
    return (p.L, p.M, p.N) if p.c_major == "n" else (p.L, p.N, p.M)


def sample_points(p: Problem, count: int, seed: int, extra=()) -> np.ndarray:
    """`count` seeded (m, n, l) points, the four corners of every batch and
    the last row/column (ragged tails) included, plus any `extra` points."""
    rng = np.random.default_rng(seed)
    pts = [rng.integers(0, p.M, count), rng.integers(0, p.N, count), rng.integers(0, p.L, count)]
    pts = np.stack(pts, axis=1)
    corners = []
    for l in range(p.L):
        for m in (0, p.M - 1):
            for n in (0, p.N - 1):
                corners.append((m, n, l))
    allp = [pts, np.array(corners, dtype=np.int64).reshape(-1, 3)]
    if len(extra):
        allp.append(np.asarray(extra, dtype=np.int64).reshape(-1, 3))
    return np.concatenate(allp, axis=0).astype(np.int64)


# ------------------------------------------------------ quantizer inputs

def real_blocks(L: int, rows: int, cols: int, seed: int, block: int = 32, spread: int = 30,
                specials: bool = False) -> np.ndarray:
    """Seeded real-valued input of the MX quantizer, float32 (L, rows, cols):
    N(0, 1) values with every `block`-element run scaled by its own 2^j,
    j uniform in [-spread, spread].  With `specials`, some runs are replaced
    by edge cases: all zeros, a NaN, an infinity, fp32 subnormals, values near
    the fp32 maximum, exact powers of two, and one value between binades."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((L, rows, cols))
    x *= np.repeat(np.exp2(rng.integers(-spread, spread + 1, (L, rows, cols // block))),
                   block, axis=2)
    x = x.astype(np.float32)
    if specials:
        nb = cols // block
        picks = rng.choice(L * rows * nb, size=min(L * rows * nb, 8), replace=False)
        for i, f in enumerate(picks):
            l, rem = divmod(int(f), rows * nb)
            r, b = divmod(rem, nb)
            blk = x[l, r, b * block:(b + 1) * block]
            kind = i % 8
            if kind == 0:
                blk[:] = 0.0
            elif kind == 1:
                blk[rng.integers(block)] = np.nan
            elif kind == 2:
                blk[rng.integers(block)] = -np.inf
            elif kind == 3:
                blk[:] = (rng.standard_normal(block) * 1e-41).astype(np.float32)
            elif kind == 4:
                blk[:] = (rng.uniform(-3.3e38, 3.3e38, block)).astype(np.float32)
            elif kind == 5:
                blk[:] = np.exp2(rng.integers(-20, 20, block)).astype(np.float32)
            elif kind == 6:
                blk[:] = 0.0
                blk[0] = -0.0
                blk[1] = 1.0e-45
            else:
                blk[:] = np.float32(1.5) * np.exp2(np.float32(rng.integers(-5, 5)))
    return x



def real_blocks_colwise(L: int, rows: int, cols: int, seed: int, block: int = 32,
                        spread: int = 30, specials: bool = False) -> np.ndarray:
    """real_blocks with the runs down the columns: float32 (L, rows, cols),
    cols contiguous, every `block` consecutive rows of a column scaled by its
    own 2^j (the input shape of the columnwise quantizer).  rows must be a
    multiple of `block`; cols is free."""
    x = real_blocks(L, cols, rows, seed, block=block, spread=spread, specials=specials)
    return np.ascontiguousarray(x.transpose(0, 2, 1))

def device_real_blocks(L: int, rows: int, cols: int, seed: int, device, block: int = 32,
                       spread: int = 30):
    """real_blocks' recipe drawn on a CUDA device by torch's seeded generator,
    for inputs too large to build on the host: N(0, 1) values, each
    `block`-element run scaled by its own 2^j, j uniform in [-spread, spread].
    Returns a float32 tensor (L, rows, cols) on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((L, rows, cols), generator=g, device=device, dtype=torch.float32)
    j = torch.randint(-spread, spread + 1, (L, rows, cols // block), generator=g, device=device)
    x.view(L, rows, cols // block, block).mul_(torch.exp2(j.float()).unsqueeze(-1))
    return x

