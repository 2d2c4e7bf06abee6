"""GPU parity of the columnwise MX quantizer (blocks of 32 down each column,
"GEMM + RoPE + MXFP8 Projection (SM100)", the S-direction) against the
oracle, through the C ABI (include/bsquant.h, direction BSG_QUANT_COLWISE):
code bytes and the whole padded scale-atom tensor bit for bit, and the
codes fed to the GEMM as MN-major operands."""
import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import oracle
import synth

pytestmark = pytest.mark.gpu

TORCH_IN = {"f32": torch.float32, "bf16": torch.bfloat16}
GUARD = 64


def run_colwise(X32: np.ndarray, in_dtype: str, out_dtype: str):
    """Kernel codes and scales for X (float32 numpy, rounded to in_dtype
    first); returns (codes, sf, exact input as float64, guards intact)."""
    Xt = torch.from_numpy(np.ascontiguousarray(X32)).to(TORCH_IN[in_dtype]).cuda()
    L, rows, cols = X32.shape
    q = bsg.make_quant_problem(rows, cols, L, in_dtype, out_dtype, 32, "col")
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


def assert_same(codes, sf, exact, out_dtype):
    ocodes, osf = oracle.quantize_colwise(exact, out_dtype, 32)
    ocodes, osf = ocodes.reshape(-1), osf.reshape(-1)
    bad = np.nonzero(codes != ocodes)[0]
    assert bad.size == 0, f"{bad.size} code bytes differ, first at {bad[:5]}: " \
                          f"gpu {codes[bad[:5]]} oracle {ocodes[bad[:5]]}"
    bad = np.nonzero(sf != osf)[0]
    assert bad.size == 0, f"{bad.size} scale bytes differ, first at {bad[:5]}: " \
                          f"gpu {sf[bad[:5]]} oracle {osf[bad[:5]]}"


# (L, rows, cols): one block, ragged atoms in both directions (rows not a
# multiple of 128, cols not a multiple of 128 or of a unit's 256 / 512
# columns), several batches, one wide and one tall case
SHAPES = [(1, 32, 16), (1, 96, 144), (2, 160, 272), (1, 128, 4096), (3, 256, 528),
          (1, 4096, 128), (2, 224, 1040)]


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("out_dtype", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"L{s[0]}x{s[1]}x{s[2]}" for s in SHAPES])
def test_parity(in_dtype, out_dtype, shape):
    L, rows, cols = shape
    X = synth.real_blocks_colwise(L, rows, cols, seed=2100 + rows + cols, block=32)
    codes, sf, exact, guards = run_colwise(X, in_dtype, out_dtype)
    assert guards, "write outside the code or scale tensor"
    assert_same(codes, sf, exact, out_dtype)


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("out_dtype", ["e4m3", "e5m2"])
def test_special_blocks(in_dtype, out_dtype):
    """Zero blocks, NaN and infinity, fp32 subnormals, values near the fp32
    maximum, powers of two, a -0 next to the smallest subnormal -- each a
    32-row run of one column."""
    X = synth.real_blocks_colwise(2, 256, 96, seed=2200, block=32, specials=True)
    codes, sf, exact, guards = run_colwise(X, in_dtype, out_dtype)
    assert guards
    assert_same(codes, sf, exact, out_dtype)


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
def test_full_size(in_dtype):
    """The measured configuration (16384 x 8192 -> E4M3), every byte."""
    X = synth.real_blocks_colwise(1, 16384, 8192, seed=2300, block=32)
    codes, sf, exact, guards = run_colwise(X, in_dtype, "e4m3")
    assert guards
    assert_same(codes, sf, exact, "e4m3")


def test_rejections_before_launch():
    q = bsg.make_quant_problem(48, 64, 1, "f32", "e4m3", 32, "col")
    assert bsg.bsg_quantize(q, 0, 0, 0, 0) == bsg.BSG_ERR_UNSUPPORTED
    q = bsg.make_quant_problem(64, 64, 1, "f32", "e2m1", 32, "col")
    assert bsg.bsg_quantize(q, 0, 0, 0, 0) == bsg.BSG_ERR_UNSUPPORTED
    x = torch.zeros(64 * 64 + 4, dtype=torch.float32, device="cuda")
    out = torch.zeros(8192, dtype=torch.uint8, device="cuda")
    q = bsg.make_quant_problem(64, 64, 1, "f32", "e4m3", 32, "col")
    st = bsg.bsg_quantize(q, x.data_ptr() + 4, out.data_ptr(), out.data_ptr() + 4096, 0)
    assert st == bsg.BSG_ERR_ALIGNMENT


@pytest.mark.parametrize("M,N,K,L", [(256, 384, 512, 1), (144, 208, 320, 2)])
def test_gemm_consumes_columnwise_operands(M, N, K, L):
    """Columnwise-quantized (K x M) and (K x N) matrices are an m-major A and
    an n-major B with their scale atoms: the GEMM on them matches the oracle
    GEMM on the same bytes (C within tolerance, Amax bit-consistent), and the
    oracle's result on the kernel's bytes is the oracle's result on its own
    columnwise quantization (the bytes are identical)."""
    import gpu_util
    At = synth.real_blocks_colwise(L, K, M, seed=2400, block=32, spread=4)
    Bt = synth.real_blocks_colwise(L, K, N, seed=2401, block=32, spread=4)
    a, sfa, ea, _ = run_colwise(At, "f32", "e4m3")
    b, sfb, eb, _ = run_colwise(Bt, "f32", "e4m3")
    oa, osa = oracle.quantize_colwise(ea, "e4m3", 32)
    assert np.array_equal(a, oa.reshape(-1)) and np.array_equal(sfa, osa.reshape(-1))
    p = synth.Problem(M=M, N=N, K=K, L=L, a_dtype="e4m3", b_dtype="e4m3", sfv=32,
                      c_dtype="bf16", c_major="n", a_major="m", b_major="n")
    inp = synth.Inputs(problem=p, A=a.reshape(L, K, M), B=b.reshape(L, K, N),
                       SFA=sfa.reshape(synth.scale_shape(M, K, 32, L)),
                       SFB=sfb.reshape(synth.scale_shape(N, K, 32, L)))
    c, amax, _, _, guard_ok = gpu_util.run_gpu(inp, guard=4096)
    assert guard_ok
    gpu_util.assert_parity(inp, c, amax)
