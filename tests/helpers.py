"""Independent numpy/torch decoding used only to pin the oracle.

Nothing here is shared with the oracle's C code: FP8 and E8M0 bytes are
decoded by torch's float8 dtypes (a library conversion), E2M1 by the value
list of the OCP MX format definition, and scales are fetched through the
6-D logical view obtained with numpy's transpose."""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# OCP Microscaling spec, FP4 E2M1 element values for codes 0..7 (sign is bit 3)
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def lib_decode(codes: np.ndarray, dtype: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    if dtype == "e4m3":
        return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if dtype == "e5m2":
        return t.view(torch.float8_e5m2).to(torch.float64).numpy()
    if dtype == "ue8m0":
        return t.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    if dtype == "e2m1":
        c = codes.astype(np.int64)
        mag = np.array(E2M1_VALUES)[c & 7]
        return np.where(c & 8, -mag, mag)
    raise KeyError(dtype)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    lo = packed & 0xF
    hi = packed >> 4
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def logical_scales(phys: np.ndarray, rows: int, kblocks: int) -> np.ndarray:
    """(L, rows, kblocks) scale bytes read through the page's logical view
    phys.transpose(3, 4, 1, 5, 2, 0) = (32, 4, T, 4, T_k, L)."""
    logical = phys.transpose(3, 4, 1, 5, 2, 0)
    r = np.arange(rows)[:, None]
    kb = np.arange(kblocks)[None, :]
    out = logical[r % 32, (r % 128) // 32, r // 128, kb % 4, kb // 4, :]  # (rows, kblocks, L)
    return np.ascontiguousarray(out.transpose(2, 0, 1))


def dense_operand(codes, dtype, phys_sf, rows, K, sfv, sf_dtype="ue8m0", major="k"):
    """Dequantized operand (L, rows, K) in float64, computed independently of the oracle.
    `codes` is k-major (L, rows, K) or, for major "m" / "n", (L, K, rows)."""
    if major != "k":
        codes = codes.reshape(-1, K, rows).transpose(0, 2, 1)
    if dtype == "e2m1":
        codes = unpack_e2m1(codes)
    vals = lib_decode(codes, dtype)
    kblocks = -(-K // sfv)
    sf = lib_decode(logical_scales(phys_sf, rows, kblocks), sf_dtype)
    return vals * np.repeat(sf, sfv, axis=2)[:, :, :K]


def independent_gemm(inp):
    p = inp.problem
    a = dense_operand(inp.A, p.a_dtype, inp.SFA, p.M, p.K, p.sfv, p.sf_dtype, p.a_major)
    b = dense_operand(inp.B, p.b_dtype, inp.SFB, p.N, p.K, p.sfv, p.sf_dtype, p.b_major)
    return np.einsum("lmk,lnk->lmn", a, b), np.einsum("lmk,lnk->lmn", np.abs(a), np.abs(b))


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def golden_names(prefix="ex"):
    """Fixture files of one kind: ``ex*`` GEMM examples, ``q*`` quantizer blocks."""
    return sorted(n for n in os.listdir(GOLDEN) if n.startswith(prefix) and n.endswith(".json"))


def build_golden_inputs(g):
    """Materialise a hand-worked fixture into synth.Inputs (codes zero, scale
    bytes 127 unless the fixture sets them)."""
    import synth
    pr = g["problem"]
    p = synth.Problem(pr["M"], pr["N"], pr["K"], pr["L"], pr["a_dtype"], pr["b_dtype"],
                      pr["sfv"], pr.get("c_dtype", "f32"), pr.get("c_major", "n"),
                      a_major=pr.get("a_major", "k"), b_major=pr.get("b_major", "k"))

    def operand(rows, dtype, fills):
        codes = np.zeros((p.L, rows, p.K), dtype=np.uint8)
        for l, r, k0, k1, code in fills:
            codes[l, r, k0:k1] = code
        if dtype == "e2m1":
            codes = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
        return codes

    def scales(rows, sets):
        kblocks = -(-p.K // p.sfv)
        sf = np.full((p.L, rows, kblocks), 127, dtype=np.uint8)
        for mn, kb, l, byte in sets:
            sf[l, mn, kb] = byte
        return synth.pack_scale_atoms(sf, rows, p.K, p.sfv)

    # a fixture may give an operand as its stored bytes, in memory order
    A = np.array(g["A_flat"], dtype=np.uint8) if "A_flat" in g else operand(p.M, p.a_dtype, g["A_fill"])
    B = np.array(g["B_flat"], dtype=np.uint8) if "B_flat" in g else operand(p.N, p.b_dtype, g["B_fill"])
    return synth.Inputs(p, A, B, scales(p.M, g["SFA_set"]), scales(p.N, g["SFB_set"]))
