"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* the library builds, loads and exports every function include/*.h declares;
* the ctypes structures have the C layout (compiled probe with gcc);
* bsg_problem_check enforces the page's support surface ("Support surface
  and constraints") and returns a status, before anything touches a device.
"""
import ctypes
import os
import re
import subprocess

import pytest

import block_scaled_precision_04_gb300 as bsg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("bsgemm.h", "bsquant.h")]


@pytest.fixture(scope="module")
def lib():
    bsg.build()
    return bsg.library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(bsg_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "bsg_run" in names and "bsg_plan_create" in names and "bsg_quantize" in names
    out = subprocess.run(["nm", "-D", "--defined-only", bsg.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (bsg_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "probe.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "bsgemm.h"
#include "bsquant.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(bsg_problem), offsetof(bsg_problem, a_major),
         offsetof(bsg_problem, sf_vec_size), offsetof(bsg_problem, cluster_n), sizeof(bsg_plan_info));
  printf("%zu %zu\n", sizeof(bsg_device_buffers), offsetof(bsg_device_buffers, ws_bytes));
  printf("%zu %zu %zu %zu\n", sizeof(bsg_quant_problem), offsetof(bsg_quant_problem, in_dtype),
         offsetof(bsg_quant_problem, sf_vec_size), offsetof(bsg_quant_problem, direction));
  return 0;
}
''')
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    a = [int(x) for x in lines[0].split()]
    b = [int(x) for x in lines[1].split()]
    assert a == [ctypes.sizeof(bsg.bsg_problem), bsg.bsg_problem.a_major.offset,
                 bsg.bsg_problem.sf_vec_size.offset, bsg.bsg_problem.cluster_n.offset,
                 ctypes.sizeof(bsg.bsg_plan_info)]
    assert b == [ctypes.sizeof(bsg.bsg_device_buffers), bsg.bsg_device_buffers.ws_bytes.offset]
    c = [int(x) for x in lines[2].split()]
    assert c == [ctypes.sizeof(bsg.bsg_quant_problem), bsg.bsg_quant_problem.in_dtype.offset,
                 bsg.bsg_quant_problem.sf_vec_size.offset, bsg.bsg_quant_problem.direction.offset]


def test_status_strings(lib):
    for s in range(8):
        assert bsg.bsg_status_string(s)
    assert bsg.bsg_status_string(0) == "ok"


OK_CASES = [
    dict(M=256, N=256, K=256, L=1),
    dict(M=4096, N=4096, K=4096, L=1, c_dtype="bf16"),
    dict(M=2048, N=2048, K=8192, L=8, a_dtype="e5m2", b_dtype="e4m3"),
    dict(M=8192, N=8192, K=8192, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16,
         c_dtype="bf16"),
    dict(M=8000, N=1000, K=7168, L=2, c_major="m"),
    dict(M=1, N=4, K=16, L=1),
    dict(M=4, N=1, K=32, L=3, c_major="m"),
    dict(M=3, N=8, K=32, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=32, c_dtype="f16"),
    dict(M=128, N=128, K=128, L=1, tile_m=128, tile_n=256, cluster_m=2, cluster_n=1),
    dict(M=256, N=256, K=256, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16,
         c_dtype="e4m3"),
    dict(M=256, N=256, K=256, L=2, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=32,
         c_dtype="e5m2", c_major="m"),
    dict(M=130, N=96, K=128, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16,
         c_dtype="e2m1"),
    dict(M=8192, N=8192, K=8192, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16,
         sf_dtype="e4m3", c_dtype="bf16"),
    dict(M=130, N=96, K=160, L=2, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16,
         sf_dtype="e4m3", c_dtype="e2m1"),
    dict(M=4096, N=4096, K=4096, L=1, a_major="m", b_major="n", c_dtype="bf16"),
    dict(M=144, N=96, K=40, L=2, a_major="m", b_major="n"),     # K free when both are MN-major
    dict(M=16, N=8, K=64, L=1, a_major="m"),
    dict(M=8, N=16, K=64, L=1, b_major="n", a_dtype="e5m2"),
    dict(M=256, N=512, K=256, L=1, b_major="n", tile_n=256, cluster_m=2),
    dict(M=256, N=512, K=256, L=1, b_major="n", tile_n=128),
    dict(M=256, N=512, K=256, L=1, a_major="m", tile_n=256, cluster_m=1),
]


@pytest.mark.parametrize("kw", OK_CASES)
def test_supported_problems_pass(lib, kw):
    assert bsg.bsg_problem_check(bsg.make_problem(**kw)) == bsg.BSG_OK


BAD_CASES = [
    # (problem, expected status, rule)
    (dict(M=0, N=4, K=32, L=1), bsg.BSG_ERR_INVALID_ARG, "empty M"),
    (dict(M=4, N=4, K=0, L=1), bsg.BSG_ERR_INVALID_ARG, "empty K"),
    (dict(M=4, N=4, K=32, L=0), bsg.BSG_ERR_INVALID_ARG, "empty L"),
    (dict(M=-1, N=4, K=32, L=1), bsg.BSG_ERR_INVALID_ARG, "negative M"),
    (dict(M=4, N=4, K=32, L=1, sf_vec_size=16), bsg.BSG_ERR_UNSUPPORTED, "FP8 with sfv 16"),
    (dict(M=4, N=4, K=32, L=1, sf_vec_size=64), bsg.BSG_ERR_INVALID_ARG, "sfv not 16/32"),
    (dict(M=4, N=4, K=32, L=1, a_dtype="e2m1", b_dtype="e4m3"), bsg.BSG_ERR_UNSUPPORTED,
     "FP4 x FP8"),
    (dict(M=4, N=4, K=32, L=1, sf_dtype="e4m3"), bsg.BSG_ERR_UNSUPPORTED,
     "E4M3 scales with FP8 operands"),
    (dict(M=4, N=4, K=64, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=32,
          sf_dtype="e4m3"), bsg.BSG_ERR_UNSUPPORTED, "E4M3 scales with sfv 32"),
    (dict(M=4, N=4, K=32, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16,
          sf_dtype="e5m2"), bsg.BSG_ERR_INVALID_ARG, "E5M2 scales"),
    (dict(M=4, N=4, K=32, L=1, sf_dtype="f32"), bsg.BSG_ERR_INVALID_ARG, "scale dtype"),
    (dict(M=4, N=4, K=32, L=1, c_dtype="e4m3"), bsg.BSG_ERR_UNSUPPORTED, "FP8 in, FP8 out"),
    (dict(M=4, N=4, K=32, L=1, c_dtype="e2m1"), bsg.BSG_ERR_UNSUPPORTED, "FP4 C with FP8 in"),
    (dict(M=4, N=64, K=64, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16, c_dtype="e2m1",
          c_major="m"), bsg.BSG_ERR_UNSUPPORTED, "FP4 C m-major"),
    (dict(M=4, N=48, K=64, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16, c_dtype="e2m1"),
     bsg.BSG_ERR_ALIGNMENT, "FP4 C row of 24 bytes"),
    (dict(M=4, N=24, K=64, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16, c_dtype="e4m3"),
     bsg.BSG_ERR_ALIGNMENT, "FP8 C row of 24 bytes"),
    (dict(M=4, N=4, K=32, L=1, c_dtype="ue8m0"), bsg.BSG_ERR_INVALID_ARG, "C dtype"),
    (dict(M=4, N=4, K=32, L=1, a_dtype="f32"), bsg.BSG_ERR_INVALID_ARG, "A dtype"),
    (dict(M=4, N=4, K=64, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16, a_major="m"),
     bsg.BSG_ERR_UNSUPPORTED, "FP4 not k-major"),
    (dict(M=4, N=4, K=32, L=1, b_major="n"), bsg.BSG_ERR_ALIGNMENT, "n-major B, N % 16"),
    (dict(M=20, N=16, K=32, L=1, a_major="m"), bsg.BSG_ERR_ALIGNMENT, "m-major A, M % 16"),
    (dict(M=16, N=16, K=40, L=1, a_major="m"), bsg.BSG_ERR_ALIGNMENT, "k-major B, K % 16"),
    (dict(M=16, N=16, K=32, L=1, a_major="n"), bsg.BSG_ERR_INVALID_ARG, "A n-major"),
    (dict(M=16, N=16, K=32, L=1, b_major="m"), bsg.BSG_ERR_INVALID_ARG, "B m-major"),
    (dict(M=16, N=16, K=64, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16, a_major="m"),
     bsg.BSG_ERR_UNSUPPORTED, "FP4 m-major"),
    (dict(M=256, N=512, K=256, L=1, tile_n=256, cluster_m=4),
     bsg.BSG_ERR_UNSUPPORTED, "cluster of four (tiles shared by multicast) not built"),
    (dict(M=256, N=512, K=256, L=1, a_major="m", tile_n=256, cluster_m=4),
     bsg.BSG_ERR_UNSUPPORTED, "cluster of four, m-major A"),
    (dict(M=256, N=512, K=256, L=1, cluster_n=2), bsg.BSG_ERR_UNSUPPORTED, "cluster along N"),
    (dict(M=256, N=512, K=256, L=1, cluster_n=4), bsg.BSG_ERR_UNSUPPORTED, "cluster of 4 along N"),
    (dict(M=256, N=512, K=256, L=1, b_major="n", tile_n=256, cluster_m=1),
     bsg.BSG_ERR_UNSUPPORTED, "n-major B 256 wide in one CTA"),
    (dict(M=4, N=4, K=32, L=1, a_major="x"), bsg.BSG_ERR_INVALID_ARG, "bad major"),
    (dict(M=4, N=4, K=32, L=1, c_major="k"), bsg.BSG_ERR_INVALID_ARG, "bad C major"),
    (dict(M=4, N=4, K=24, L=1), bsg.BSG_ERR_ALIGNMENT, "FP8 row of 24 bytes"),
    (dict(M=4, N=4, K=48, L=1, a_dtype="e2m1", b_dtype="e2m1", sf_vec_size=16),
     bsg.BSG_ERR_ALIGNMENT, "FP4 row of 24 bytes"),
    (dict(M=4, N=6, K=32, L=1), bsg.BSG_ERR_ALIGNMENT, "fp32 C row of 24 bytes"),
    (dict(M=4, N=12, K=32, L=1, c_dtype="bf16"), bsg.BSG_ERR_ALIGNMENT, "bf16 C row of 24 B"),
    (dict(M=6, N=8, K=32, L=1, c_major="m"), bsg.BSG_ERR_ALIGNMENT, "m-major C column 24 B"),
    (dict(M=4, N=4, K=32, L=1, tile_m=256), bsg.BSG_ERR_INVALID_ARG, "TILE_M 256 disabled"),
    (dict(M=4, N=4, K=32, L=1, tile_n=64), bsg.BSG_ERR_INVALID_ARG, "TILE_N 64"),
    (dict(M=4, N=4, K=32, L=1, cluster_m=3), bsg.BSG_ERR_INVALID_ARG, "cluster 3"),
    (dict(M=1 << 31, N=4, K=32, L=1), bsg.BSG_ERR_INVALID_ARG, "M beyond 2^31-1"),
]


@pytest.mark.parametrize("kw,status,rule", BAD_CASES, ids=[c[2] for c in BAD_CASES])
def test_support_surface_rejections(lib, kw, status, rule):
    assert bsg.bsg_problem_check(bsg.make_problem(**kw)) == status, rule


def test_null_problem_rejected(lib):
    assert lib.bsg_problem_check(None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.bsg_plan_create(None, 0, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.bsg_plan_workspace_size(None, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.bsg_run(None, None, None, None, None, None, None, None, 0, None) == \
        bsg.BSG_ERR_INVALID_ARG
    lib.bsg_plan_destroy(None)


def test_plan_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    st, plan = bsg.bsg_plan_create(bsg.make_problem(256, 256, 256, 1), 0)
    assert st in (bsg.BSG_ERR_CUDA, bsg.BSG_ERR_ARCH)
    assert not plan.value


def test_invalid_problem_fails_before_device(lib):
    """Validation happens first: an unsupported problem is reported as such
    even on a machine with no GPU."""
    st, _ = bsg.bsg_plan_create(bsg.make_problem(4, 4, 32, 1, sf_vec_size=16), 0)
    assert st == bsg.BSG_ERR_UNSUPPORTED


QUANT_OK = [
    dict(rows=1, cols=32),
    dict(rows=16384, cols=8192, in_dtype="bf16", out_dtype="e2m1", sf_vec_size=16),
    dict(rows=130, cols=96, L=3, out_dtype="e5m2"),
    dict(rows=7, cols=64, out_dtype="e2m1", sf_vec_size=32),
    dict(rows=32, cols=16, direction="col"),
    dict(rows=16384, cols=8192, in_dtype="bf16", out_dtype="e5m2", direction="col"),
    dict(rows=96, cols=144, L=3, direction="col"),
]


@pytest.mark.parametrize("kw", QUANT_OK)
def test_quant_supported(lib, kw):
    assert bsg.bsg_quant_check(bsg.make_quant_problem(**kw)) == bsg.BSG_OK


QUANT_BAD = [
    (dict(rows=0, cols=32), bsg.BSG_ERR_INVALID_ARG, "empty rows"),
    (dict(rows=4, cols=0), bsg.BSG_ERR_INVALID_ARG, "empty cols"),
    (dict(rows=4, cols=32, L=0), bsg.BSG_ERR_INVALID_ARG, "empty L"),
    (dict(rows=1 << 20, cols=32, L=1 << 12), bsg.BSG_ERR_INVALID_ARG, "rows * L beyond 2^31-1"),
    (dict(rows=4, cols=32, in_dtype="f16"), bsg.BSG_ERR_INVALID_ARG, "fp16 input"),
    (dict(rows=4, cols=32, out_dtype="bf16"), bsg.BSG_ERR_INVALID_ARG, "bf16 output"),
    (dict(rows=4, cols=32, sf_vec_size=64), bsg.BSG_ERR_INVALID_ARG, "sfv 64"),
    (dict(rows=4, cols=32, out_dtype="e4m3", sf_vec_size=16), bsg.BSG_ERR_UNSUPPORTED, "FP8 sfv 16"),
    (dict(rows=4, cols=48), bsg.BSG_ERR_UNSUPPORTED, "partial block"),
    (dict(rows=4, cols=32, direction=2), bsg.BSG_ERR_INVALID_ARG, "unknown direction"),
    (dict(rows=64, cols=32, out_dtype="e2m1", sf_vec_size=32, direction="col"),
     bsg.BSG_ERR_UNSUPPORTED, "columnwise E2M1"),
    (dict(rows=64, cols=32, out_dtype="e2m1", sf_vec_size=16, direction="col"),
     bsg.BSG_ERR_UNSUPPORTED, "columnwise sfv 16"),
    (dict(rows=48, cols=32, direction="col"), bsg.BSG_ERR_UNSUPPORTED, "columnwise partial block"),
    (dict(rows=64, cols=24, direction="col"), bsg.BSG_ERR_ALIGNMENT, "columnwise row of 24 B"),
    (dict(rows=64, cols=32, in_dtype="f16", direction="col"), bsg.BSG_ERR_INVALID_ARG,
     "columnwise fp16 input"),
]


@pytest.mark.parametrize("kw,status,rule", QUANT_BAD, ids=[c[2] for c in QUANT_BAD])
def test_quant_rejections(lib, kw, status, rule):
    assert bsg.bsg_quant_check(bsg.make_quant_problem(**kw)) == status, rule


def test_quant_sizes(lib):
    st, (cb, sb) = bsg.bsg_quant_sizes(bsg.make_quant_problem(130, 256, 2, "bf16", "e2m1", 16))
    assert st == bsg.BSG_OK and cb == 2 * 130 * 128 and sb == 2 * 2 * 4 * 512
    assert lib.bsg_quantize(None, None, None, None, None) == bsg.BSG_ERR_INVALID_ARG
    # columnwise: codes in X's layout; atoms over ceil(cols/128) x ceil(rows/128)
    st, (cb, sb) = bsg.bsg_quant_sizes(bsg.make_quant_problem(160, 272, 2, "f32", "e4m3", 32, "col"))
    assert st == bsg.BSG_OK and cb == 2 * 160 * 272 and sb == 2 * 3 * 2 * 512



def test_problem_bytes_match_the_layouts():
    """The tensor sizes the Python wrapper checks before a launch: codes
    (packed E2M1 two per byte), whole scale atoms, and C of its dtype."""
    pb = bsg.problem_bytes(bsg.make_problem(300, 200, 96, 2, "e4m3", "e5m2", 32, "bf16"))
    assert pb == {"A": 2 * 300 * 96, "B": 2 * 200 * 96, "SFA": 2 * 3 * 1 * 512,
                  "SFB": 2 * 2 * 1 * 512, "C": 2 * 300 * 200 * 2}
    pb = bsg.problem_bytes(bsg.make_problem(130, 96, 128, 1, "e2m1", "e2m1", 16, "e2m1"))
    assert pb == {"A": 130 * 64, "B": 96 * 64, "SFA": 2 * 2 * 512, "SFB": 1 * 2 * 512,
                  "C": 130 * 48}
    # every synthetic generator's tensors have exactly these sizes
    import synth
    p = synth.Problem(300, 200, 96, 2, "e4m3", "e5m2", 32, "bf16")
    inp = synth.uniform_codes(p, 3)
    pb = bsg.problem_bytes(bsg.make_problem(300, 200, 96, 2, "e4m3", "e5m2", 32, "bf16"))
    assert (inp.A.nbytes, inp.B.nbytes, inp.SFA.nbytes, inp.SFB.nbytes) == \
        (pb["A"], pb["B"], pb["SFA"], pb["SFB"])
