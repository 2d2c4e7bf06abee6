"""GPU parity of the MX quantizer (csrc/quant.cu) against the oracle, through
the C ABI (include/bsquant.h): code bytes and the whole padded scale-atom
tensor must match bit for bit.  Both sides decide each code from x / 2^e with
a power-of-two e, so the same value is rounded (exactly representable
in the kernel's fp32 except below fp32's normal range, where every format
rounds to zero)."""
import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import oracle
import synth

pytestmark = pytest.mark.gpu

TORCH_IN = {"f32": torch.float32, "bf16": torch.bfloat16}
GUARD = 64


def run_gpu(X32: np.ndarray, in_dtype: str, out_dtype: str, sfv: int):
    """Kernel codes and scales for X (float32 numpy, rounded to in_dtype first);
    returns (codes, sf, exact input as float64, guards intact)."""
    Xt = torch.from_numpy(np.ascontiguousarray(X32)).to(TORCH_IN[in_dtype]).cuda()
    L, rows, cols = X32.shape
    q = bsg.make_quant_problem(rows, cols, L, in_dtype, out_dtype, sfv)
    st, (cb, sb) = bsg.bsg_quant_sizes(q)
    assert st == bsg.BSG_OK
    cbuf = torch.full((cb + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    sbuf = torch.full((sb + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    codes, sf = cbuf[GUARD:GUARD + cb], sbuf[GUARD:GUARD + sb]
    st = bsg.bsg_quantize(q, Xt.data_ptr(), codes.data_ptr(), sf.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    assert st == bsg.BSG_OK, bsg.bsg_status_string(st)
    torch.cuda.synchronize()
    guards = bool((cbuf[:GUARD] == 0xA5).all() and (cbuf[GUARD + cb:] == 0xA5).all()
                  and (sbuf[:GUARD] == 0xA5).all() and (sbuf[GUARD + sb:] == 0xA5).all())
    exact = Xt.float().cpu().numpy().astype(np.float64)
    return codes.cpu().numpy(), sf.cpu().numpy(), exact, guards


def assert_same(codes, sf, exact, out_dtype, sfv):
    ocodes, osf = oracle.quantize(exact, out_dtype, sfv)
    ocodes, osf = ocodes.reshape(-1), osf.reshape(-1)
    bad = np.nonzero(codes != ocodes)[0]
    assert bad.size == 0, f"{bad.size} code bytes differ, first at {bad[:5]}: " \
                          f"gpu {codes[bad[:5]]} oracle {ocodes[bad[:5]]}"
    bad = np.nonzero(sf != osf)[0]
    assert bad.size == 0, f"{bad.size} scale bytes differ, first at {bad[:5]}: " \
                          f"gpu {sf[bad[:5]]} oracle {osf[bad[:5]]}"


FORMATS = [("e4m3", 32), ("e5m2", 32), ("e2m1", 16), ("e2m1", 32)]
SHAPES = [(1, 1, 32), (1, 130, 96), (2, 37, 256), (1, 128, 4096), (3, 200, 160), (1, 3, 2048)]


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("out_dtype,sfv", FORMATS)
@pytest.mark.parametrize("shape", SHAPES)
def test_parity(in_dtype, out_dtype, sfv, shape):
    L, rows, cols = shape
    if cols % sfv:
        pytest.skip("whole blocks only")
    X = synth.real_blocks(L, rows, cols, seed=1100 + rows + cols, block=sfv)
    codes, sf, exact, guards = run_gpu(X, in_dtype, out_dtype, sfv)
    assert guards, "write outside the code or scale tensor"
    assert_same(codes, sf, exact, out_dtype, sfv)


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("out_dtype,sfv", FORMATS)
def test_special_blocks(in_dtype, out_dtype, sfv):
    """Zero blocks, NaN and infinity, fp32 subnormals, values near the fp32
    maximum, powers of two, a -0 next to the smallest subnormal."""
    X = synth.real_blocks(2, 65, 8 * sfv, seed=1200, block=sfv, specials=True)
    codes, sf, exact, guards = run_gpu(X, in_dtype, out_dtype, sfv)
    assert guards
    assert_same(codes, sf, exact, out_dtype, sfv)


@pytest.mark.parametrize("in_dtype,out_dtype,sfv", [("f32", "e4m3", 32), ("bf16", "e2m1", 16)])
def test_full_size_sampled(in_dtype, out_dtype, sfv):
    """The measured configuration (16384 x 8192), checked on sampled rows."""
    rows, cols = 16384, 8192
    X = synth.real_blocks(1, rows, cols, seed=1300, block=sfv)
    codes, sf, exact, guards = run_gpu(X, in_dtype, out_dtype, sfv)
    assert guards
    rng = np.random.default_rng(5)
    pick = np.unique(np.concatenate([[0, 127, 128, rows - 1], rng.integers(0, rows, 60)]))
    per_row = cols // 2 if out_dtype == "e2m1" else cols
    c = codes.reshape(rows, per_row)
    t_k = -(-(cols // sfv) // 4)
    for r in pick:
        oc, osf = oracle.quantize(exact[:, r:r + 1, :], out_dtype, sfv)
        assert np.array_equal(c[r], oc.reshape(-1)), r
        for b in range(cols // sfv):
            got = sf[oracle.sf_offset(int(r), b, 0, -(-rows // 128), t_k)]
            want = osf.reshape(-1)[oracle.sf_offset(0, b, 0, 1, t_k)]
            assert got == want, (r, b)


def test_rejections_before_launch():
    q = bsg.make_quant_problem(4, 48, 1, "f32", "e4m3", 32)
    assert bsg.bsg_quantize(q, 0, 0, 0, 0) == bsg.BSG_ERR_UNSUPPORTED
    x = torch.zeros(4 * 64 + 1, dtype=torch.float32, device="cuda")
    q = bsg.make_quant_problem(4, 64, 1, "f32", "e4m3", 32)
    out = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    st = bsg.bsg_quantize(q, x.data_ptr() + 4, out.data_ptr(), out.data_ptr() + 1024, 0)
    assert st == bsg.BSG_ERR_ALIGNMENT


def test_gemm_consumes_kernel_quantized_operands():
    """Operands quantized by this kernel feed the GEMM: its result matches the
    oracle GEMM on the same codes and scales (the formats line up)."""
    import gpu_util
    M, N, K = 256, 192, 512
    XA = synth.real_blocks(1, M, K, seed=1400, block=32, spread=4)
    XB = synth.real_blocks(1, N, K, seed=1401, block=32, spread=4)
    a, sfa, _, _ = run_gpu(XA, "f32", "e4m3", 32)
    b, sfb, _, _ = run_gpu(XB, "f32", "e4m3", 32)
    p = synth.Problem(M=M, N=N, K=K, L=1, a_dtype="e4m3", b_dtype="e4m3", sfv=32,
                      c_dtype="f32", c_major="n")
    inp = synth.Inputs(problem=p, A=a.reshape(1, M, K), B=b.reshape(1, N, K),
                       SFA=sfa.reshape(synth.scale_shape(M, K, 32, 1)),
                       SFB=sfb.reshape(synth.scale_shape(N, K, 32, 1)))
    c, amax, _, _, _ = gpu_util.run_gpu(inp)
    gpu_util.assert_parity(inp, c, amax)
