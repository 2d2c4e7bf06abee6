"""Parity at sizes past 32-bit element counts: a C of more than 2^32 elements
(one batch, and three batches whose offsets pass 2^32 bytes) and a quantizer
input of more than 2^31 elements.  These are the widest tensors the library
indexes; they are checked at sampled points against the oracle, with Amax
compared with the maximum of the whole C taken on the device."""
import numpy as np
import pytest
import torch

import block_scaled_precision_04_gb300 as bsg
import oracle
import synth
from gpu_util import TORCH_C, problem_of, to_device

pytestmark = pytest.mark.gpu


def _gemm_sampled(p: synth.Problem, seed: int):
    inp = synth.uniform_codes(p, seed, 122, 130)
    op = bsg.GemmAmax(problem_of(p))
    A, B, SFA, SFB = to_device(inp)
    C = torch.empty(synth.c_shape(p), dtype=TORCH_C[p.c_dtype], device="cuda:0")
    amax = torch.full((1,), -1.0, dtype=torch.float32, device="cuda:0")
    op.run(A, B, SFA, SFB, C, amax)
    torch.cuda.synchronize()
    assert op.device_status() == bsg.BSG_OK
    # Amax: the largest |C| over every stored element, bit for bit
    whole = C.float().abs().amax().item()
    assert np.float32(amax.item()).view(np.uint32) == np.float32(whole).view(np.uint32)
    extra = [(p.M - 1, p.N - 1, p.L - 1), (p.M // 2, p.N - 1, p.L - 1), (p.M - 1, 0, 0)]
    pts = synth.sample_points(p, 2048, seed + 1, extra)
    # element (m, n, l) of an n-major C sits at flat index (l*M + m)*N + n
    flat = torch.from_numpy((pts[:, 2] * p.M + pts[:, 0]) * p.N + pts[:, 1]).cuda()
    got = C.view(-1).index_select(0, flat).float().cpu().numpy().astype(np.float64)
    cref, s = oracle.gemm_sample(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B,
                                 inp.SFA, inp.SFB, pts)
    cref = oracle.round_to(cref, p.c_dtype)
    tau = oracle.tolerance(cref, s, p.c_dtype)
    bad = ~(np.abs(got - cref) <= tau)
    assert not bad.any(), [(tuple(pts[i]), got[i], cref[i]) for i in np.flatnonzero(bad)[:8]]


def test_gemm_c_past_2_32_elements():
    """65600 x 65552 bf16 C: 4.3e9 elements, 8.6 GB; the far corners sit past
    2^32 elements."""
    _gemm_sampled(synth.Problem(65600, 65552, 128, 1, "e4m3", "e4m3", 32, "bf16", "n"), 71)


def test_gemm_batches_past_2_32_bytes():
    """Three 40000 x 40000 fp32 batches: 4.8e9 elements, 19.2 GB; the batch
    offsets pass 2^32 bytes."""
    _gemm_sampled(synth.Problem(40000, 40000, 64, 3, "e5m2", "e4m3", 32, "f32", "n"), 73)


def test_quantize_input_past_2_31_elements():
    """70000 x 32768 fp32 input (2.3e9 elements, 9.2 GB) to E4M3: sampled rows,
    the last included, byte for byte against the oracle."""
    rows, cols, sfv = 70000, 32768, 32
    X = synth.device_real_blocks(1, rows, cols, 77, "cuda:0", block=sfv)
    codes, sf = bsg.quantize(X, "e4m3", sfv)
    torch.cuda.synchronize()
    t_r, t_k = -(-rows // 128), -(-(cols // sfv) // 4)
    rng = np.random.default_rng(78)
    for r in np.unique(np.concatenate([[0, 65535, 65536, rows - 1], rng.integers(0, rows, 12)])):
        x = X[0, int(r)].cpu().numpy().astype(np.float64)[None, None, :]
        oc, osf = oracle.quantize(x, "e4m3", sfv)
        got = codes[int(r) * cols:(int(r) + 1) * cols].cpu().numpy()
        assert np.array_equal(got, oc.reshape(-1)), int(r)
        offs = torch.tensor([oracle.sf_offset(int(r), b, 0, t_r, t_k) for b in range(cols // sfv)],
                            device="cuda:0")
        got_sf = sf.index_select(0, offs).cpu().numpy()
        want_sf = np.array([osf.reshape(-1)[oracle.sf_offset(0, b, 0, 1, t_k)]
                            for b in range(cols // sfv)], dtype=np.uint8)
        assert np.array_equal(got_sf, want_sf), int(r)
