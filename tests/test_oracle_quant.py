"""Pins of the oracle's MX quantizer (the row upstream of the GEMM) to things
other than itself.

* **Hand-worked blocks** (``tests/golden/q*.json``): each with its citation
  and derivation.
* **Element rounding:** against torch's float8 conversions of float32 values,
  which round to nearest even; E2M1 against an exhaustive grid worked with
  exact fractions.
* **Defining properties:**
  - the block maximum lands in the element format's top binade;
  - the rounding error stays within half a step of the element format;
  - negating the input flips only the sign bits;
  - scaling by 2^j moves only the scale bytes;
  - an already-quantized tensor with a top-binade element in every block
    round-trips exactly through the pinned dequantizer;
  - special blocks and atom padding behave as stated.
* **A third implementation:** the input generator's numpy/torch quantizer,
  on ordinary data.

No GPU needed.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import E2M1_VALUES, golden_names

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EMAX = {"e4m3": 8, "e5m2": 15, "e2m1": 2}
MAXV = {"e4m3": 448.0, "e5m2": 57344.0, "e2m1": 6.0}
SIGN = {"e4m3": 0x80, "e5m2": 0x80, "e2m1": 0x8}


def code_at(codes, dtype, l, r, k):
    if dtype == "e2m1":
        b = int(codes[l, r, k // 2])
        return b & 0xF if k % 2 == 0 else b >> 4
    return int(codes[l, r, k])


def unpack(codes, dtype):
    """Codes as one integer per element, shape (L, rows, cols)."""
    if dtype != "e2m1":
        return codes.astype(np.int64)
    lo = (codes & 0xF).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    out = np.empty(codes.shape[:2] + (codes.shape[2] * 2,), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def scale_bytes(sf, rows, nblk):
    """Scale bytes as (L, rows, nblk), through the pinned atom offsets."""
    L, t_r, t_k = sf.shape[:3]
    flat = sf.reshape(-1)
    out = np.empty((L, rows, nblk), dtype=np.int64)
    for l in range(L):
        for r in range(rows):
            for b in range(nblk):
                out[l, r, b] = flat[oracle.sf_offset(r, b, l, t_r, t_k)]
    return out


@pytest.mark.parametrize("name", golden_names("q"))
def test_golden_blocks(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    X = np.zeros((1, g["rows"], g["cols"]))
    for k, v in g.get("x_set", []):
        X[0, 0, k] = v
    for r, k, v in g.get("x_set_rc", []):
        X[0, r, k] = v
    codes, sf = oracle.quantize(X, g["out_dtype"], g["sfv"])
    for k, v in g.get("expect_codes", []):
        assert code_at(codes, g["out_dtype"], 0, 0, k) == v, (name, k)
    for r, k, v in g.get("expect_codes_rc", []):
        assert code_at(codes, g["out_dtype"], 0, r, k) == v, (name, r, k)
    t_r, t_k = sf.shape[1], sf.shape[2]
    for r, b, v in g["expect_scale_bytes"]:
        assert int(sf.reshape(-1)[oracle.sf_offset(r, b, 0, t_r, t_k)]) == v, (name, r, b)


@pytest.mark.parametrize("name", golden_names("cq"))
def test_golden_columnwise_blocks(name):
    """Hand-worked columnwise blocks (blocks of 32 down each column)."""
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    X = np.zeros((1, g["rows"], g["cols"]))
    for r, c, v in g["x_set_rc"]:
        X[0, r, c] = float(v)
    codes, sf = oracle.quantize_colwise(X, g["out_dtype"], g["sfv"])
    for r, c, v in g["expect_codes_rc"]:
        assert int(codes[0, r, c]) == v, (name, r, c)
    t_c, t_k = sf.shape[1], sf.shape[2]
    flat = sf.reshape(-1)
    seen = set()
    for c, b, v in g["expect_scale_bytes"]:
        off = oracle.sf_offset(c, b, 0, t_c, t_k)
        seen.add(off)
        assert int(flat[off]) == v, (name, c, b)
    rest = np.array([flat[i] for i in range(flat.size) if i not in seen])
    assert np.all(rest == g["expect_padding_byte"])


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2"])
@pytest.mark.parametrize("L,rows,cols", [(1, 32, 16), (2, 96, 48), (1, 160, 272), (3, 256, 130)])
def test_columnwise_is_rowwise_of_the_transpose(dtype, L, rows, cols):
    """Blocks down the columns of X are blocks along the rows of X^T: the
    columnwise codes are the rowwise codes of X^T transposed back, and the
    scale of (column c, block b) is the rowwise scale of (row c, block b) --
    the same atom tensor byte for byte, padding included.  Ragged shapes
    (rows not a multiple of 128, cols not a multiple of 128) and special
    blocks are included."""
    X = synth.real_blocks_colwise(L, rows, cols, seed=rows + cols + L, block=32)
    X = X.astype(np.float64)
    X[0, 0:32, 0] = 0.0                           # a zero block
    X[L - 1, rows - 32 + 5, cols - 1] = np.nan    # a NaN block in the last corner
    if cols > 2:
        X[0, 32 % rows, 1] = np.inf
    cc, sc = oracle.quantize_colwise(X, dtype, 32)
    cr, sr = oracle.quantize(np.ascontiguousarray(X.transpose(0, 2, 1)), dtype, 32)
    np.testing.assert_array_equal(cc, cr.transpose(0, 2, 1))
    np.testing.assert_array_equal(sc, sr)


def test_columnwise_block_properties():
    """Each column block's maximum lands in the top binade of E4M3 (its code
    is 0x78..0x7E in magnitude), and no code of a block exceeds it."""
    X = synth.real_blocks_colwise(1, 128, 64, seed=5, block=32).astype(np.float64)
    X = X * np.exp2(np.random.default_rng(6).integers(-20, 20, size=(1, 1, 64)))  # columns differ
    codes, sf = oracle.quantize_colwise(X, "e4m3", 32)
    for c in range(64):
        for b in range(4):
            col = codes[0, 32 * b:32 * b + 32, c].astype(np.int64) & 0x7F
            blk = X[0, 32 * b:32 * b + 32, c]
            top = col[np.argmax(np.abs(blk))]
            assert 0x78 <= top <= 0x7E, (c, b, top)
            assert col.max() == top


@pytest.mark.parametrize("bad", [dict(dtype="e2m1"), dict(sfv=16), dict(rows=48)])
def test_columnwise_rejects(bad):
    rows = bad.get("rows", 64)
    X = np.ones((1, rows, 16))
    with pytest.raises(ValueError):
        oracle.quantize_colwise(X, bad.get("dtype", "e4m3"), bad.get("sfv", 32))


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2"])
def test_columnwise_quantize_then_mn_major_gemm_within_the_formats_error(dtype):
    """A (K x M) and B (K x N) stored with M (N) contiguous, quantized
    columnwise (blocks of 32 along K), are an m-major A and an n-major B
    with their scale atoms; the GEMM oracle on them gives the product of the
    original matrices within the error the two quantisations allow (the
    bound of the rowwise test, with blocks along K).  A scale keyed by the
    wrong column or block, or codes read as k-major, break it."""
    M, N, K, L = 144, 200, 320, 2
    At = synth.real_blocks_colwise(L, K, M, seed=51, block=32).astype(np.float64)  # (L, K, M)
    Bt = synth.real_blocks_colwise(L, K, N, seed=52, block=32).astype(np.float64)
    At *= np.exp2(np.random.default_rng(53).integers(-6, 6, size=(L, 1, M)))
    qa, sa = oracle.quantize_colwise(At, dtype, 32)
    qb, sb = oracle.quantize_colwise(Bt, dtype, 32)
    C, _, _ = oracle.gemm(M, N, K, L, dtype, dtype, 32, qa, qb, sa, sb, a_major="m", b_major="n")
    rel, ab = ERR[dtype]

    def err(Xt):  # Xt (L, K, MN): blocks of 32 along K
        Lx, Kx, MNx = Xt.shape
        blk = np.abs(Xt).reshape(Lx, Kx // 32, 32, MNx)
        bm = blk.max(axis=2, keepdims=True)
        unit = np.where(bm > 0, 2.0 ** (np.floor(np.log2(np.where(bm > 0, bm, 1.0))) - EMAX[dtype]), 0.0)
        return (rel * blk + ab * unit).reshape(Xt.shape)

    ea, eb = err(At), err(Bt)
    exact = np.einsum("lkm,lkn->lmn", At, Bt)
    bound = (np.einsum("lkm,lkn->lmn", np.abs(At), eb) + np.einsum("lkm,lkn->lmn", ea, np.abs(Bt)) +
             np.einsum("lkm,lkn->lmn", ea, eb))
    assert np.all(np.abs(C - exact) <= bound * (1 + 1e-12) + 1e-300)
    assert np.median(np.abs(C - exact) / np.maximum(bound, 1e-300)) < 0.5
    # the same bytes read as k-major, or A's scales of the two column atoms
    # swapped, break the bound
    Cw, _, _ = oracle.gemm(M, N, K, L, dtype, dtype, 32,
                           np.ascontiguousarray(qa.reshape(L, M, K)),
                           np.ascontiguousarray(qb.reshape(L, N, K)), sa, sb)
    assert not np.all(np.abs(Cw - exact) <= bound * (1 + 1e-12))
    sa_swapped = np.ascontiguousarray(sa[:, ::-1])
    Cs, _, _ = oracle.gemm(M, N, K, L, dtype, dtype, 32, qa, qb, sa_swapped, sb,
                           a_major="m", b_major="n")
    assert not np.all(np.abs(Cs - exact) <= bound * (1 + 1e-12))


@pytest.mark.parametrize("dtype,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_element_rounding_matches_torch(dtype, tdt):
    rng = np.random.default_rng(7)
    m = MAXV[dtype]
    # float32 inputs (torch then rounds once), spread over every binade in range
    mag = np.exp2(rng.uniform(-20, np.log2(m), 20000)).astype(np.float32)
    y = (mag * rng.choice([-1, 1], mag.size)).astype(np.float32)
    y = y[np.abs(y) <= m]
    # exact ties: midpoints between neighbouring codes
    tab = oracle.decode_table(dtype)
    finite = [c for c in range(0x80) if np.isfinite(tab[c])]
    mids = np.array([(tab[c] + tab[c + 1]) / 2 for c in finite[:-1]], dtype=np.float64)
    mids = mids[mids.astype(np.float32) == mids].astype(np.float32)
    y = np.concatenate([y, mids, -mids, np.float32([0.0, -0.0, m, -m])])
    want = torch.from_numpy(y).to(tdt).view(torch.uint8).numpy()
    got = np.array([oracle.quantize_value(float(v), dtype) for v in y], dtype=np.uint8)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["e4m3", "e5m2", "e2m1"])
def test_saturation(dtype):
    m = MAXV[dtype]
    maxc = oracle.quantize_value(m, dtype)
    for y in (m * 1.01, m * 1.5, m * 8, 1e30):
        assert oracle.quantize_value(y, dtype) == maxc
        assert oracle.quantize_value(-y, dtype) == maxc | SIGN[dtype]


def test_e2m1_exhaustive_grid():
    vals = [Fraction(v).limit_denominator(4) for v in E2M1_VALUES[:8]]  # 0 .. 6, codes 0 .. 7
    for i in range(-8 * 64, 8 * 64 + 1):
        y = Fraction(i, 64)
        a = abs(y)
        if a >= vals[-1]:
            c = 7
        else:
            best = min(range(8), key=lambda c: (abs(vals[c] - a), c & 1))
            c = best
        if y < 0 or (y == 0 and i < 0):
            c |= 0x8
        assert oracle.quantize_value(float(y), "e2m1") == c, float(y)


def random_blocks(rng, L, rows, cols, sfv):
    # magnitudes spread over many binades, per block
    x = rng.standard_normal((L, rows, cols))
    x *= np.repeat(np.exp2(rng.integers(-30, 30, (L, rows, cols // sfv))), sfv, axis=2)
    return x.astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype,sfv", [("e4m3", 32), ("e5m2", 32), ("e2m1", 16), ("e2m1", 32)])
def test_block_properties(dtype, sfv):
    rng = np.random.default_rng(11)
    L, rows, cols = 2, 37, 4 * sfv
    X = random_blocks(rng, L, rows, cols, sfv)
    codes, sf = oracle.quantize(X, dtype, sfv)
    c = unpack(codes, dtype)
    sb = scale_bytes(sf, rows, cols // sfv)
    tab = oracle.decode_table(dtype)
    dec = tab[c]
    scale = np.exp2(sb.astype(np.float64) - 127).repeat(sfv, axis=2)
    y = X / scale
    # the block maximum lands in the top binade [2^emax, 2^(emax+1))
    ymax = np.abs(y).reshape(L, rows, -1, sfv).max(axis=3)
    assert np.all(ymax >= 2.0 ** EMAX[dtype]) and np.all(ymax < 2.0 ** (EMAX[dtype] + 1))
    # rounding error: within half the spacing of the format at |y|, or saturated
    m = MAXV[dtype]
    mant = {"e4m3": 3, "e5m2": 2, "e2m1": 1}[dtype]
    emin = {"e4m3": -6, "e5m2": -14, "e2m1": 0}[dtype]
    ay = np.abs(y)
    ex = np.maximum(np.floor(np.log2(np.where(ay > 0, ay, 1.0))), emin)
    half = np.exp2(ex - mant) / 2
    sat = ay > m
    assert np.all(np.abs(dec[~sat] - y[~sat]) <= half[~sat])
    assert np.all(np.abs(dec[sat]) == m) and np.all(np.sign(dec[sat]) == np.sign(y[sat]))


@pytest.mark.parametrize("dtype,sfv", [("e4m3", 32), ("e5m2", 32), ("e2m1", 16)])
def test_sign_and_power_of_two_invariance(dtype, sfv):
    rng = np.random.default_rng(5)
    X = random_blocks(rng, 1, 9, 2 * sfv, sfv)
    codes, sf = oracle.quantize(X, dtype, sfv)
    ncodes, nsf = oracle.quantize(-X, dtype, sfv)
    assert np.array_equal(unpack(ncodes, dtype), unpack(codes, dtype) ^ SIGN[dtype])
    assert np.array_equal(nsf, sf)
    for j in (-3, 1, 7):
        scodes, ssf = oracle.quantize(X * 2.0 ** j, dtype, sfv)
        assert np.array_equal(scodes, codes)
        a = scale_bytes(sf, 9, 2).astype(np.int64)
        b = scale_bytes(ssf, 9, 2).astype(np.int64)
        assert np.array_equal(b - a, np.full_like(a, j))


@pytest.mark.parametrize("dtype,sfv", [("e4m3", 32), ("e5m2", 32), ("e2m1", 16), ("e2m1", 32)])
def test_exact_round_trip_of_mx_data(dtype, sfv):
    """Codes with one top-binade element per block and finite scales,
    dequantized by the pinned GEMM-side dequantizer, quantize back to
    themselves."""
    rng = np.random.default_rng(3)
    L, rows, cols = 1, 130, 8 * sfv
    tab = oracle.decode_table(dtype)
    finite = np.array([c for c in range(len(tab)) if np.isfinite(tab[c])])
    top = np.array([c for c in finite if 2.0 ** EMAX[dtype] <= abs(tab[c]) <= MAXV[dtype]])
    c = rng.choice(finite, (L, rows, cols))
    c[..., ::sfv] = rng.choice(top, (L, rows, cols // sfv))
    if dtype == "e2m1":
        packed = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    else:
        packed = c.astype(np.uint8)
    sfl = rng.integers(100, 150, (L, rows, cols // sfv)).astype(np.uint8)
    sf = synth.pack_scale_atoms(sfl, rows, cols, sfv)
    X = oracle.dequantize(packed, dtype, sf, sfv, rows, cols, L)
    codes, sf2 = oracle.quantize(X, dtype, sfv)
    got = unpack(codes, dtype)
    want = c.copy()
    # a zero keeps its sign bit through dequantize/quantize
    assert np.array_equal(got, want)
    assert np.array_equal(sf2, sf)


def test_special_blocks_and_padding():
    X = np.zeros((1, 3, 64))
    X[0, 1, 5] = np.nan
    X[0, 2, 40] = np.inf
    X[0, 2, 2] = 1.0
    codes, sf = oracle.quantize(X, "e4m3", 32)
    sb = scale_bytes(sf, 3, 2)
    assert sb[0, 0, 0] == 127 and sb[0, 0, 1] == 127          # all-zero blocks
    assert sb[0, 1, 0] == 0xFF and np.all(codes[0, 1, :32] == 0x7F)
    assert sb[0, 1, 1] == 127 and np.all(codes[0, 1, 32:] == 0)
    assert sb[0, 2, 1] == 0xFF and np.all(codes[0, 2, 32:] == 0x7F)
    assert sb[0, 2, 0] == 127 - 8 and codes[0, 2, 2] == 0x78   # 1.0 -> 256 = 2^8
    # every other byte of the padded atom (rows 3..127, blocks 2..3) is 127
    flat = sf.reshape(-1)
    used = {oracle.sf_offset(r, b, 0, 1, 1) for r in range(3) for b in range(2)}
    assert all(flat[i] == 127 for i in range(flat.size) if i not in used)


@pytest.mark.parametrize("dtype,sfv", [("e4m3", 32), ("e5m2", 32), ("e2m1", 16)])
def test_matches_the_input_generator(dtype, sfv):
    """The seeded generators carry their own quantizer (numpy frexp, float32
    scaling, torch casts); on ordinary data both follow the same rule."""
    rng = np.random.default_rng(17)
    x = rng.standard_normal((64, 8 * sfv)).astype(np.float32)
    codes_g, sf_g = synth.quantize_blocks(x, dtype, sfv)
    codes_o, sf_o = oracle.quantize(x.astype(np.float64)[None], dtype, sfv)
    assert np.array_equal(codes_o[0], codes_g)
    assert np.array_equal(scale_bytes(sf_o, 64, 8)[0], sf_g.astype(np.int64))


# ------------------------------------------------- low-precision C rounding

@pytest.mark.parametrize("dtype,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_c_rounding_matches_torch_saturated(dtype, tdt):
    """C rounded to FP8: round to nearest even with saturation, i.e. torch's
    (round-to-nearest-even) cast of the value clamped to the largest finite
    magnitude, decoded back."""
    rng = np.random.default_rng(23)
    m = MAXV[dtype]
    x = (np.exp2(rng.uniform(-24, np.log2(m) + 3, 20000)) *
         rng.choice([-1, 1], 20000)).astype(np.float32)
    want = torch.from_numpy(np.clip(x, -m, m)).to(tdt).to(torch.float64).numpy()
    got = oracle.round_to(x.astype(np.float64), dtype)
    assert np.array_equal(got, want)


def test_c_rounding_e2m1_grid_and_specials():
    vals = [Fraction(v).limit_denominator(4) for v in E2M1_VALUES[:8]]
    ys = [Fraction(i, 64) for i in range(-9 * 64, 9 * 64 + 1)]
    got = oracle.round_to(np.array([float(y) for y in ys]), "e2m1")
    for y, g in zip(ys, got):
        a = abs(y)
        c = 7 if a >= vals[-1] else min(range(8), key=lambda c: (abs(vals[c] - a), c & 1))
        want = float(vals[c]) * (-1.0 if y < 0 else 1.0)
        assert g == want, float(y)
    spec = oracle.round_to(np.array([np.nan, np.inf, -np.inf]), "e2m1")
    assert spec[0] == 0.0 and spec[1] == 6.0 and spec[2] == -6.0
    spec = oracle.round_to(np.array([np.nan, np.inf, -np.inf, 1e30]), "e4m3")
    assert np.isnan(spec[0]) and list(spec[1:]) == [448.0, -448.0, 448.0]


@pytest.mark.parametrize("dtype,spacing_at_1,emax", [("e4m3", 0.125, 8), ("e5m2", 0.25, 15),
                                                     ("e2m1", 0.5, 2)])
def test_c_ulp(dtype, spacing_at_1, emax):
    """The tolerance's ulp: the gap between neighbouring codes at |x|, taken
    from the decode table (capped at the largest binade)."""
    assert oracle.ulp(1.0, dtype) == spacing_at_1
    tab = np.sort(np.unique(np.abs(oracle.decode_table(dtype)[np.isfinite(oracle.decode_table(dtype))])))
    for lo, hi in zip(tab[1:-1], tab[2:]):
        if lo >= 2.0 ** (emax - 3):   # normal range: the spacing right above lo
            assert oracle.ulp(lo, dtype) == hi - lo or lo >= 2.0 ** emax
    assert oracle.ulp(tab[-1] * 4, dtype) == oracle.ulp(tab[-1], dtype)


# per-element error of one MX quantisation, from the formats alone: at most
# REL |x| (saturation of the top binade, or half a step relative to the value)
# plus ABS 2^e (half the subnormal step, in the block's scale 2^e)
ERR = {"e4m3": (0.125, 2.0 ** -10), "e5m2": (0.125, 2.0 ** -17), "e2m1": (0.25, 0.25)}


@pytest.mark.parametrize("dtype,sfv", [("e4m3", 32), ("e5m2", 32), ("e2m1", 32), ("e2m1", 16)])
def test_quantize_then_gemm_within_the_formats_error(dtype, sfv):
    """The quantizer's codes and scale atoms, read back by the GEMM oracle,
    give the product of the original real matrices within the error the two
    quantisations allow: |C - A B^T| <= sum_k |a| eb + ea |b| + ea eb, with
    e = REL |x| + ABS 2^(floor(log2 blockmax) - emax).  A scale written to the
    wrong atom position, row or K block, or a wrong binade, breaks it."""
    M, N, K, L = 200, 136, 384, 2
    A = synth.real_blocks(L, M, K, seed=41, block=sfv).astype(np.float64)
    B = synth.real_blocks(L, N, K, seed=42, block=sfv).astype(np.float64)
    qa, sa = oracle.quantize(A, dtype, sfv)
    qb, sb = oracle.quantize(B, dtype, sfv)
    C, _, _ = oracle.gemm(M, N, K, L, dtype, dtype, sfv, qa, qb, sa, sb)
    rel, ab = ERR[dtype]

    def err(X):
        bm = np.abs(X).reshape(L, X.shape[1], K // sfv, sfv).max(axis=-1, keepdims=True)
        unit = np.where(bm > 0, 2.0 ** (np.floor(np.log2(np.where(bm > 0, bm, 1.0))) - EMAX[dtype]), 0.0)
        return (rel * np.abs(X).reshape(bm.shape[:-1] + (sfv,)) + ab * unit).reshape(X.shape)

    ea, eb = err(A), err(B)
    exact = np.einsum("lmk,lnk->lmn", A, B)
    bound = (np.einsum("lmk,lnk->lmn", np.abs(A), eb) + np.einsum("lmk,lnk->lmn", ea, np.abs(B)) +
             np.einsum("lmk,lnk->lmn", ea, eb))
    assert np.all(np.abs(C - exact) <= bound * (1 + 1e-12) + 1e-300)
    # and the bound is not vacuous: the quantised product is close in bulk
    assert np.median(np.abs(C - exact) / np.maximum(bound, 1e-300)) < 0.5
