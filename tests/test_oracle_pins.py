"""Pins of the CPU oracle to facts outside itself.

Each test checks the oracle against something the pages or the mathematics
fix: hand-worked examples (tests/golden), library decodes of the number
formats, the page's layout permutation, closed forms, scale-factor
invariants and brute force through an independent numpy path.  A plausible
slip in the oracle (a dropped term, a wrong sign, a transposed operand, a
swapped atom index) fails at least one of them.
"""
import fractions
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (E2M1_VALUES, build_golden_inputs, dense_operand, golden_names,
                     independent_gemm, lib_decode, load_golden, logical_scales)


def run_oracle(inp, **kw):
    p = inp.problem
    kw.setdefault("sf_dtype", p.sf_dtype)
    kw.setdefault("a_major", p.a_major)
    kw.setdefault("b_major", p.b_major)
    return oracle.gemm(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                       inp.SFA, inp.SFB, **kw)


# ----------------------------------------------------------------- decoding

@pytest.mark.parametrize("dtype", ["e4m3", "e5m2", "ue8m0"])
def test_decode_table_matches_torch(dtype):
    """Every 8-bit code decodes as torch's float8 dtypes do (a library routine)."""
    ours = oracle.decode_table(dtype)
    ref = lib_decode(np.arange(256, dtype=np.uint8), dtype)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.where(both_nan, 0, ours), np.where(both_nan, 0, ref))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_decode_e2m1_matches_ocp_value_list():
    ours = oracle.decode_table("e2m1")
    expect = np.array(E2M1_VALUES + [-v for v in E2M1_VALUES])
    assert np.array_equal(ours, expect)


def test_decode_special_values():
    e4m3 = oracle.decode_table("e4m3")
    assert e4m3[0x38] == 1.0 and e4m3[0x40] == 2.0 and e4m3[0xB8] == -1.0
    assert e4m3[0x7E] == 448.0 and e4m3[0xFE] == -448.0
    assert e4m3[0x01] == 2.0 ** -9 and e4m3[0x08] == 2.0 ** -6
    assert math.isnan(e4m3[0x7F]) and math.isnan(e4m3[0xFF])
    assert np.sum(np.isnan(e4m3)) == 2
    e5m2 = oracle.decode_table("e5m2")
    assert e5m2[0x3C] == 1.0 and e5m2[0x7B] == 57344.0
    assert e5m2[0x7C] == math.inf and e5m2[0xFC] == -math.inf
    assert math.isnan(e5m2[0x7D]) and e5m2[0x01] == 2.0 ** -16 and e5m2[0x04] == 2.0 ** -14
    e8 = oracle.decode_table("ue8m0")
    assert e8[127] == 1.0 and e8[0] == 2.0 ** -127 and e8[254] == 2.0 ** 127
    assert math.isnan(e8[255])


# ------------------------------------------------------------ atom layout

@pytest.mark.parametrize("seed", range(6))
def test_sf_offset_is_the_pages_permutation(seed):
    """The oracle's direct offset names the same byte as the page's logical
    view: physical (L, T, T_k, 32, 4, 4) permuted by (3, 4, 1, 5, 2, 0)."""
    rng = np.random.default_rng(seed)
    L, T, TK = rng.integers(1, 4), rng.integers(1, 5), rng.integers(1, 5)
    phys = np.arange(L * T * TK * 512).reshape(L, T, TK, 32, 4, 4)
    logical = phys.transpose(3, 4, 1, 5, 2, 0)
    assert logical.shape == (32, 4, T, 4, TK, L)
    for _ in range(200):
        m0, m1, mt = rng.integers(32), rng.integers(4), rng.integers(T)
        kin, kt, l = rng.integers(4), rng.integers(TK), rng.integers(L)
        mn = 128 * mt + 32 * m1 + m0
        kb = 4 * kt + kin
        assert oracle.sf_offset(mn, kb, l, T, TK) == logical[m0, m1, mt, kin, kt, l]


def test_generator_atoms_agree_with_oracle_offsets():
    """synth.pack_scale_atoms (numpy reshapes) and the oracle's offset
    formula (arithmetic) are written independently; they must agree."""
    rng = np.random.default_rng(7)
    L, rows, K, sfv = 2, 200, 320, 32
    kblocks = K // sfv
    sf = rng.integers(0, 256, size=(L, rows, kblocks)).astype(np.uint8)
    phys = synth.pack_scale_atoms(sf, rows, K, sfv).reshape(-1)
    T, TK = -(-rows // 128), -(-K // (4 * sfv))
    for l in range(L):
        for r in range(rows):
            for kb in range(kblocks):
                assert phys[oracle.sf_offset(r, kb, l, T, TK)] == sf[l, r, kb]


# ------------------------------------------------------ hand-worked examples

@pytest.mark.parametrize("name", golden_names())
def test_golden_example(name):
    g = load_golden(name)
    pr = g["problem"]
    for mn, kb, l, off in g.get("expect_sf_offset", []):
        T, TK = -(-pr["M"] // 128), -(-pr["K"] // (4 * pr["sfv"]))
        assert oracle.sf_offset(mn, kb, l, T, TK) == off, (mn, kb, l)
    inp = build_golden_inputs(g)
    p = inp.problem
    ref = oracle.reference(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                           inp.SFA, inp.SFB, p.c_dtype, a_major=p.a_major, b_major=p.b_major)
    for m, n, l, v in g["expect_C"]:
        assert ref["exact"][l, m, n] == v, (m, n, l)
        assert ref["c"][l, m, n] == v
    assert ref["amax"] == g["expect_amax"]


# ------------------------------------------------------------- invariants

def _small(seed, a="e4m3", b="e4m3", sfv=32, M=40, N=24, K=128, L=2, lo=124, hi=130):
    p = synth.Problem(M, N, K, L, a, b, sfv, "f32", "n")
    return synth.uniform_codes(p, seed, lo, hi)


def test_unit_scales_reduce_to_plain_gemm():
    """All scale bytes 127 (2^0): C is the plain GEMM of the decoded codes
    (the page's own JAX example uses np.ones scales)."""
    inp = _small(11, lo=127, hi=127)
    p = inp.problem
    C, _, _ = run_oracle(inp)
    a = lib_decode(inp.A, "e4m3")
    b = lib_decode(inp.B, "e4m3")
    plain = np.stack([a[l] @ b[l].T for l in range(p.L)])
    np.testing.assert_array_equal(C, plain)


def test_the_pages_usage_example():
    """The example of "GEMM + Amax (SM100)", section "Using JAX arrays": m=512,
    n=256, k=256, sf_vec_size 32, E5M2 operands made by casting standard
    normal draws (here torch's float8_e5m2 cast of a seeded draw), every scale
    1.0 (E8M0 byte 127) in the physical atom shape (1, m/128, k/128, 32, 4, 4),
    fp32 C.  With unit scales the result is the plain product of the decoded
    operands; E5M2 products and their 256-term sums are exact in double, so
    the two agree bit for bit."""
    m, n, k, sfv = 512, 256, 256, 32
    g = torch.Generator().manual_seed(512)
    A = torch.randn(1, m, k, generator=g).to(torch.float8_e5m2).view(torch.uint8).numpy()
    B = torch.randn(1, n, k, generator=g).to(torch.float8_e5m2).view(torch.uint8).numpy()
    SFA = np.full((1, m // 128, k // (4 * sfv), 32, 4, 4), 127, dtype=np.uint8)
    SFB = np.full((1, n // 128, k // (4 * sfv), 32, 4, 4), 127, dtype=np.uint8)
    C, _, _ = oracle.gemm(m, n, k, 1, "e5m2", "e5m2", sfv, A, B, SFA, SFB)
    a, b = lib_decode(A, "e5m2")[0], lib_decode(B, "e5m2")[0]
    np.testing.assert_array_equal(C[0], a @ b.T)
    ref = oracle.reference(m, n, k, 1, "e5m2", "e5m2", sfv, A, B, SFA, SFB, "f32")
    assert ref["amax"] == np.abs(np.float32(a @ b.T)).max()


def test_one_scale_step_doubles_exactly_one_block():
    """Raising one scale byte by one doubles exactly that (row, K-block)
    term: C' - C equals the block's partial dot product (to double rounding)."""
    inp = _small(12)
    p = inp.problem
    C0, _, _ = run_oracle(inp)
    m, kb, l = 33, 2, 1
    sfa = inp.SFA.copy().reshape(-1)
    T, TK = p.t_m, p.t_k
    sfa[oracle.sf_offset(m, kb, l, T, TK)] += 1
    inp2 = synth.Inputs(p, inp.A, inp.B, sfa.reshape(inp.SFA.shape), inp.SFB)
    C1, _, _ = run_oracle(inp2)
    diff = C1 - C0
    assert np.all(diff[:, np.arange(p.M) != m, :] == 0)
    assert np.all(diff[1 - l] == 0)
    a = dense_operand(inp.A, "e4m3", inp.SFA, p.M, p.K, p.sfv)
    b = dense_operand(inp.B, "e4m3", inp.SFB, p.N, p.K, p.sfv)
    ks = slice(kb * p.sfv, (kb + 1) * p.sfv)
    block = a[l, m, ks] @ b[l, :, ks].T
    np.testing.assert_allclose(diff[l, m, :], block, rtol=0, atol=1e-12 * np.abs(block).max())


def test_row_scale_shift_scales_row():
    """Adding d to every scale byte of row m multiplies row m of C by 2^d."""
    inp = _small(13)
    p = inp.problem
    C0, _, _ = run_oracle(inp)
    m, d = 5, 3
    sfa = inp.SFA.copy().reshape(-1)
    for l in range(p.L):
        for kb in range(p.K // p.sfv):
            sfa[oracle.sf_offset(m, kb, l, p.t_m, p.t_k)] += d
    C1, _, _ = run_oracle(synth.Inputs(p, inp.A, inp.B, sfa.reshape(inp.SFA.shape), inp.SFB))
    np.testing.assert_array_equal(C1[:, m, :], C0[:, m, :] * 2.0 ** d)
    others = np.arange(p.M) != m
    np.testing.assert_array_equal(C1[:, others, :], C0[:, others, :])


def test_batches_are_independent():
    inp = _small(14, L=3)
    p = inp.problem
    C, _, _ = run_oracle(inp)
    for l in range(p.L):
        q = synth.Problem(p.M, p.N, p.K, 1, p.a_dtype, p.b_dtype, p.sfv)
        one = synth.Inputs(q, inp.A[l:l + 1], inp.B[l:l + 1], inp.SFA[l:l + 1], inp.SFB[l:l + 1])
        C1, _, _ = run_oracle(one)
        np.testing.assert_array_equal(C1[0], C[l])


def test_operands_not_transposed():
    """C[m, n] pairs row m of A with row n of B: swapping A and B transposes C."""
    inp = _small(15, M=24, N=40)
    p = inp.problem
    C, _, _ = run_oracle(inp)
    q = synth.Problem(p.N, p.M, p.K, p.L, p.b_dtype, p.a_dtype, p.sfv)
    C2, _, _ = run_oracle(synth.Inputs(q, inp.B, inp.A, inp.SFB, inp.SFA))
    np.testing.assert_array_equal(C2, C.transpose(0, 2, 1))


# ------------------------------------------------------------- brute force

@pytest.mark.parametrize("a,b,sfv", [("e4m3", "e4m3", 32), ("e5m2", "e4m3", 32),
                                     ("e5m2", "e5m2", 32), ("e2m1", "e2m1", 16),
                                     ("e2m1", "e2m1", 32)])
@pytest.mark.parametrize("K", [16, 32, 64, 96])
def test_brute_force_tiny(a, b, sfv, K):
    """All M, N <= 3, L <= 2 against the independent numpy path."""
    rng = np.random.default_rng(K * 7 + sfv)
    for M in (1, 2, 3):
        for N in (1, 2, 3):
            for L in (1, 2):
                p = synth.Problem(M, N, K, L, a, b, sfv, "f32", "n")
                inp = synth.uniform_codes(p, int(rng.integers(1 << 30)), 120, 134)
                C, S, _ = run_oracle(inp)
                Ci, Si = independent_gemm(inp)
                scale = np.maximum(Si, 1e-300)
                assert np.all(np.abs(C - Ci) <= 1e-15 * scale), (M, N, L)
                np.testing.assert_allclose(S, Si, rtol=1e-15, atol=0)


def test_e2m1_exhaustive_pairs():
    """Every E2M1 code against every E2M1 code with a few scales: C equals
    the product of the two listed values times the two scales."""
    codes = np.arange(16, dtype=np.uint8)
    M = N = 16
    K = 32
    p = synth.Problem(M, N, K, 1, "e2m1", "e2m1", 16, "f32", "n")
    A = np.zeros((1, M, K), dtype=np.uint8)
    B = np.zeros((1, N, K), dtype=np.uint8)
    A[0, :, 0] = codes  # element 0 of each row; the rest is code 0
    B[0, :, 0] = codes
    pack = lambda x: (x[..., 0::2] | (x[..., 1::2] << 4)).astype(np.uint8)
    for sa, sb in [(127, 127), (125, 130), (140, 110)]:
        sfa = np.full((1, M, 2), sa, dtype=np.uint8)
        sfb = np.full((1, N, 2), sb, dtype=np.uint8)
        inp = synth.Inputs(p, pack(A), pack(B), synth.pack_scale_atoms(sfa, M, K, 16),
                           synth.pack_scale_atoms(sfb, N, K, 16))
        C, _, _ = run_oracle(inp)
        vals = np.array(E2M1_VALUES + [-v for v in E2M1_VALUES])
        expect = np.outer(vals, vals) * 2.0 ** (sa - 127) * 2.0 ** (sb - 127)
        np.testing.assert_array_equal(C[0], expect)


# ------------------------------------------------------ E4M3 (NVFP4) scales

# A few E4M3 bytes with their values worked out by hand from the format
# (bias 7, three mantissa bits, exponent field 0 subnormal with 2^-6 * m/8).
E4M3_SCALE_BYTES = {0x38: 1.0, 0x3C: 1.5, 0x30: 0.5, 0x40: 2.0, 0x45: 3.25,
                    0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x7E: 448.0}


def test_e4m3_scale_exhaustive_pairs():
    """Every E2M1 code against every E2M1 code under hand-decoded E4M3 scales
    (sfv 16): C is the product of the two listed values and the two scales."""
    codes = np.arange(16, dtype=np.uint8)
    M = N = 16
    K = 32
    p = synth.Problem(M, N, K, 1, "e2m1", "e2m1", 16, "f32", "n", sf_dtype="e4m3")
    A = np.zeros((1, M, K), dtype=np.uint8)
    B = np.zeros((1, N, K), dtype=np.uint8)
    A[0, :, 17] = codes  # element 17: the second K-block of each row
    B[0, :, 17] = codes
    pack = lambda x: (x[..., 0::2] | (x[..., 1::2] << 4)).astype(np.uint8)
    vals = np.array(E2M1_VALUES + [-v for v in E2M1_VALUES])
    for sa, sb in [(0x38, 0x38), (0x3C, 0x45), (0x01, 0x7E), (0x07, 0x08), (0x30, 0x40)]:
        sfa = np.full((1, M, 2), 0x38, dtype=np.uint8)
        sfb = np.full((1, N, 2), 0x38, dtype=np.uint8)
        sfa[..., 1] = sa  # only the second block's scale matters
        sfb[..., 1] = sb
        inp = synth.Inputs(p, pack(A), pack(B),
                           synth.pack_scale_atoms(sfa, M, K, 16, synth.E4M3_ONE),
                           synth.pack_scale_atoms(sfb, N, K, 16, synth.E4M3_ONE))
        C, S, _ = run_oracle(inp)
        expect = np.outer(vals, vals) * E4M3_SCALE_BYTES[sa] * E4M3_SCALE_BYTES[sb]
        np.testing.assert_array_equal(C[0], expect)
        np.testing.assert_array_equal(S[0], np.abs(expect))


@pytest.mark.parametrize("K", [16, 48, 160])
@pytest.mark.parametrize("lo,hi", [(0x28, 0x50), (0x01, 0x0F), (0x60, 0x7E)])
def test_e4m3_scale_brute_force_tiny(K, lo, hi):
    """Random E4M3 scale bytes (normal, subnormal, near the top) with sfv 16
    against the independent numpy path, whose scales are decoded by torch."""
    rng = np.random.default_rng(K + lo)
    for M, N, L in [(1, 1, 1), (3, 2, 2), (5, 7, 1)]:
        p = synth.Problem(M, N, K, L, "e2m1", "e2m1", 16, "f32", "n", sf_dtype="e4m3")
        inp = synth.uniform_codes(p, int(rng.integers(1 << 30)), lo, hi)
        C, S, _ = run_oracle(inp)
        Ci, Si = independent_gemm(inp)
        assert np.all(np.abs(C - Ci) <= 1e-15 * np.maximum(Si, 1e-300)), (M, N, L)
        np.testing.assert_allclose(S, Si, rtol=1e-15, atol=0)


def test_e4m3_scale_differs_from_e8m0_reading():
    """The same scale bytes read as E4M3 and as E8M0 give different C (a
    scale-table mix-up would pass the E8M0 pins but fail here)."""
    p8 = synth.Problem(4, 4, 32, 1, "e2m1", "e2m1", 16, "f32", "n")
    inp = synth.uniform_codes(p8, 5, 0x38, 0x38)
    C8, _, _ = run_oracle(inp)
    C4, _, _ = run_oracle(inp, sf_dtype="e4m3")
    np.testing.assert_array_equal(C4, C8 * 2.0 ** (2 * (127 - 0x38)))


# ------------------------------------------------------- MN-major operands

@pytest.mark.parametrize("am,bm", [("m", "k"), ("k", "n"), ("m", "n")])
@pytest.mark.parametrize("a,b", [("e4m3", "e4m3"), ("e5m2", "e4m3")])
def test_mn_major_brute_force(am, bm, a, b):
    """m-major A / n-major B ("Parameters": strides (1, M, M*K)) against the
    independent numpy path, which transposes the stored bytes itself."""
    rng = np.random.default_rng(len(am + bm + a + b))
    for M, N, K, L in [(1, 1, 32, 1), (3, 2, 64, 2), (5, 7, 96, 1), (16, 32, 40, 2)]:
        p = synth.Problem(M, N, K, L, a, b, 32, "f32", "n", a_major=am, b_major=bm)
        inp = synth.uniform_codes(p, int(rng.integers(1 << 30)), 120, 134)
        assert inp.A.shape == ((L, K, M) if am == "m" else (L, M, K))
        C, S, _ = run_oracle(inp)
        Ci, Si = independent_gemm(inp)
        assert np.all(np.abs(C - Ci) <= 1e-15 * np.maximum(Si, 1e-300)), (M, N, K, L)
        np.testing.assert_allclose(S, Si, rtol=1e-15, atol=0)


def test_mn_major_is_a_relayout_only():
    """The same logical operands stored k-major and MN-major give the same C
    bit for bit (the oracle sums in the same order either way)."""
    p = synth.Problem(24, 40, 160, 2, "e4m3", "e5m2", 32, "f32", "n")
    inp = synth.uniform_codes(p, 77, 118, 136)
    C0, S0, _ = run_oracle(inp)
    q = synth.Problem(24, 40, 160, 2, "e4m3", "e5m2", 32, "f32", "n", a_major="m", b_major="n")
    inq = synth.Inputs(q, np.ascontiguousarray(inp.A.transpose(0, 2, 1)),
                       np.ascontiguousarray(inp.B.transpose(0, 2, 1)), inp.SFA, inp.SFB)
    C1, S1, _ = run_oracle(inq)
    np.testing.assert_array_equal(C0, C1)
    np.testing.assert_array_equal(S0, S1)
    # and reading MN-major bytes as k-major gives something else
    C2, _, _ = run_oracle(inq, a_major="k", b_major="k")
    assert not np.array_equal(C0, C2)


def test_mn_major_fp4_rejected():
    p = synth.Problem(4, 4, 32, 1, "e2m1", "e2m1", 16, "f32", "n")
    inp = synth.uniform_codes(p, 1)
    with pytest.raises(ValueError):
        run_oracle(inp, a_major="m")


# -------------------------------------------------------------- closed form

def test_uniform_code_workload_against_exact_rationals():
    """On the uniform-code workload (the 256^3 case at reduced M, N) every
    decoded value and product is a dyadic rational; the oracle's double sum
    equals the exact rational sum within the double summation bound
    K * 2^-53 * sum |terms|."""
    inp = synth.workload(1, M=6, N=5)
    p = inp.problem
    C, S, _ = run_oracle(inp)
    a = lib_decode(inp.A, "e4m3")
    b = lib_decode(inp.B, "e4m3")
    kblocks = p.K // p.sfv
    sfa = lib_decode(logical_scales(inp.SFA, p.M, kblocks), "ue8m0")
    sfb = lib_decode(logical_scales(inp.SFB, p.N, kblocks), "ue8m0")
    F = fractions.Fraction
    for m in range(p.M):
        for n in range(p.N):
            exact = sum(F(float(a[0, m, k])) * F(float(sfa[0, m, k // p.sfv]))
                        * F(float(b[0, n, k])) * F(float(sfb[0, n, k // p.sfv]))
                        for k in range(p.K))
            err = abs(F(float(C[0, m, n])) - exact)
            assert err <= F(p.K) * F(2) ** -53 * F(float(S[0, m, n]))


# ------------------------------------------------------ rounding, tolerance

def test_round_to_f32_matches_ieee_cast():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 39, 20000),
                        [0.0, -0.0, 1e-46, 3.4028235677973366e38, 3.5e38, -3.5e38]])
    with np.errstate(over="ignore"):  # the overflow to infinity is part of the check
        want = x.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(oracle.round_to(x, "f32"), want)


def test_round_to_f16_matches_numpy_half():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 5, 20000),
                        [65504.0, 65519.99, 65520.0, -70000.0, 2.0 ** -25, 2.0 ** -24 * 1.5]])
    with np.errstate(over="ignore"):  # the overflow to infinity is part of the check
        want = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(oracle.round_to(x, "f16"), want)


def test_round_to_bf16_matches_torch():
    """torch's float32 -> bfloat16 conversion rounds to nearest even; on
    float32-representable inputs the oracle's double -> bf16 rounding must agree."""
    rng = np.random.default_rng(5)
    x32 = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3.3895e38],
                    dtype=np.float32)
    x32 = np.concatenate([x32, ties])
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_to(x32.astype(np.float64), "bf16"), ref)
    assert oracle.round_to(np.array([1.0 + 2.0 ** -8]), "bf16")[0] == 1.0
    assert oracle.round_to(np.array([1.0 + 3 * 2.0 ** -8]), "bf16")[0] == 1.0 + 2.0 ** -6


def test_ulp_values():
    assert oracle.ulp(1.0, "f32") == 2.0 ** -23
    assert oracle.ulp(1.5, "bf16") == 2.0 ** -7
    assert oracle.ulp(1.0, "f16") == 2.0 ** -10
    assert oracle.ulp(0.0, "f32") == 2.0 ** -149
    assert oracle.ulp(65504.0, "f16") == 32.0
    xs = np.array([1e-3, 0.7, 3.0, 1e5, 1e30])
    for x in xs:
        assert oracle.ulp(x, "f32") == float(np.spacing(np.float32(x)))
        assert oracle.ulp(-x, "f32") == float(np.spacing(np.float32(x)))


def test_tolerance_formula():
    cref = np.array([1.0, -3.0, 0.0])
    S = np.array([100.0, 10.0, 0.0])
    tau = oracle.tolerance(cref, S, "bf16")
    np.testing.assert_array_equal(tau, [1e-3 + 2.0 ** -7, 1e-4 + 2.0 ** -6, 2.0 ** -133])


SAMPLE_CASES = [
    synth.Problem(130, 70, 96, 2, "e5m2", "e4m3", 32, "f32", "n"),
    synth.Problem(144, 80, 72, 2, "e4m3", "e5m2", 32, "f32", "n", a_major="m", b_major="n"),
    synth.Problem(48, 136, 64, 1, "e4m3", "e4m3", 32, "f32", "n", a_major="m"),
    synth.Problem(130, 70, 96, 2, "e2m1", "e2m1", 16, "f32", "n", sf_dtype="e4m3"),
]


@pytest.mark.parametrize("p", SAMPLE_CASES, ids=lambda p: f"{p.a_dtype}-{p.a_major}{p.b_major}-{p.sf_dtype}")
def test_sample_matches_full(p):
    """The point-by-point form gives the full form's sums bit for bit, for
    every operand layout and scale type the full form takes."""
    lo, hi = (0x30, 0x40) if p.sf_dtype == "e4m3" else (124, 130)
    inp = synth.uniform_codes(p, 16, lo, hi)
    C, S, _ = run_oracle(inp)
    pts = synth.sample_points(p, 300, 1)
    c, s = oracle.gemm_sample(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                              inp.SFA, inp.SFB, pts, sf_dtype=p.sf_dtype, a_major=p.a_major,
                              b_major=p.b_major)
    np.testing.assert_array_equal(c, C[pts[:, 2], pts[:, 0], pts[:, 1]])
    np.testing.assert_array_equal(s, S[pts[:, 2], pts[:, 0], pts[:, 1]])


def test_row_range_matches_full():
    inp = _small(17, M=70)
    p = inp.problem
    C, S, _ = run_oracle(inp)
    Cr, Sr, _ = run_oracle(inp, rows=(20, 51))
    np.testing.assert_array_equal(Cr, C[:, 20:51])
    np.testing.assert_array_equal(Sr, S[:, 20:51])


def test_threads_do_not_change_results():
    inp = _small(18, M=64)
    C1, _, n1 = run_oracle(inp, nthreads=1)
    C4, _, n4 = run_oracle(inp, nthreads=4)
    assert n1 == 1 and n4 == 4
    np.testing.assert_array_equal(C1, C4)
