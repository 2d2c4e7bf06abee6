"""Benchmark of the block-scaled GEMM + Amax on GB300.

One step = one launch of the whole hot path (operand/scale loads, block-scaled
MMA, epilogue with the fused Amax) over one batch of seeded synthetic input
of the chosen workload (default: MXFP8 4096^3, bf16 C).  Metric: TFLOP/s =
2*M*N*K*L / kernel time (CUDA events on the launching stream), L2 flushed
between steps.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample
  python bench.py --op quantize [--qworkload 1..4]  # the MX quantizer (HBM GB/s);
                                                    # 3, 4: columnwise blocks

Under torchrun (N > 1) the ranks share one problem, one process per GPU
(block_scaled_precision_04_gb300.shard): by default (--shard batches) the
workload's batches are repeated N times and every rank computes its own L of
them -- fixed work per GPU, "weak" scaling; --shard rows splits the workload
itself by 128-row scale atoms -- fixed total work, "strong" scaling.  The one
exchange, the 4-byte max of the per-rank Amax over NCCL, is inside every timed
step.  `--gpus N` without torchrun re-launches this script under
torch.distributed.run with N processes; under torchrun it must equal
WORLD_SIZE.  Rank 0 prints the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "block-scaled GEMM+amax TFLOP/s on 1 GB300; % of FP8/FP4 dense tensor peak"
L2_FLUSH_BYTES = 512 << 20  # > 4x the 129 MB L2
L2_NOTE = ("flushed between timed steps: a 512 MiB buffer written, then read, so the "
           "timed step starts with no input in L2 and no dirty lines to write back")


def flush_l2(buf) -> None:
    """Evict L2 outside the timed region: write a buffer larger than L2, then
    read it so that the written lines are retired to HBM before the next
    timed step rather than during it."""
    buf.zero_()
    buf.amax()
NOMINAL_RATIO = {"fp8": 4.5 / 2.25, "fp4": 13.5 / 2.25}  # dense tensor peak vs bf16
# Block-scaled MMA throughput per SM and clock, measured on GB300 with
# back-to-back tcgen05.mma (M=128 or a 256-row CTA pair, N=256): FP8 8192
# FMA, FP4 (mxf4nvf4 2X/4X, mxf4) 16384 FMA -- twice FP8, not the nominal 3x
MEASURED_FP4_OVER_FP8 = 2.0
FALLBACK_BF16_TFLOPS = 1900.0
# DRAM bytes per launch of the GEMM kernel from an ncu capture, keyed by the
# kernel source it was taken on (sha256 prefix of csrc/bsgemm.cu with its
# comments and whitespace removed, so only a code change invalidates an
# entry) and workload.
TRAFFIC = {
    ("c4e10b47e5246bc0", 1): 183552,
    ("c4e10b47e5246bc0", 2): 35740416,
    ("c4e10b47e5246bc0", 3): 415345920,
    ("c4e10b47e5246bc0", 4): 201296896,
    ("c4e10b47e5246bc0", 5): 190004224,
    ("c4e10b47e5246bc0", 6): 201825792,
    ("c4e10b47e5246bc0", 7): 35858944,
}


# the same for the quantizer kernel (csrc/quant.cu), keyed by its code hash
# and quantizer workload.  An HBM-bound kernel's writes partly stay in L2 when
# it ends (up to the 129 MB L2), so its write bytes read below the codes and
# scales it writes.
TRAFFIC_Q = {
    ("0f77d477e8d11bf4", 1): 624514304,
    ("0f77d477e8d11bf4", 2): 289173504,
    ("0f77d477e8d11bf4", 3): 625460224,
    ("0f77d477e8d11bf4", 4): 374182144,
}

QMETRIC = "MX quantize GB/s on 1 GB300 (X read + codes and scales written); % of HBM copy bandwidth"
# name, rows, cols, input dtype, code dtype, sf_vec_size, direction ("row":
# blocks along each row; "col": blocks of 32 down each column, the page's
# S-direction, whose codes are the GEMM's MN-major operand)
QWORKLOADS = {
    1: ("quantize-f32-16384x8192-e4m3-sfv32", 16384, 8192, "f32", "e4m3", 32, "row"),
    2: ("quantize-bf16-16384x8192-e2m1-sfv16", 16384, 8192, "bf16", "e2m1", 16, "row"),
    3: ("quantize-colwise-f32-16384x8192-e4m3-sfv32", 16384, 8192, "f32", "e4m3", 32, "col"),
    4: ("quantize-colwise-bf16-16384x8192-e4m3-sfv32", 16384, 8192, "bf16", "e4m3", 32, "col"),
}


def kernel_source_hash(name: str = "bsgemm.cu") -> str:
    import re
    path = os.path.join(ROOT, "block_scaled_precision_04_gb300", "csrc", name)
    with open(path) as f:
        src = f.read()
    # drop comments (string literals in this file hold no comment markers)
    # and all whitespace
    code = re.sub(r"//[^\n]*|/\*.*?\*/", "", src, flags=re.S)
    code = re.sub(r"\s+", "", code)
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank sets the time)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, total_ms: float) -> float:
    """Work of every replica (one per rank) over the slowest rank's time."""
    return world * flops_per_step * steps / (total_ms / 1e3) / 1e12


def batch_seed(number: int, rank: int) -> int:
    """Seed of the batches rank `rank` owns in a batch-sharded run: rank 0's
    are the workload itself (seed 1000 + number), every other rank's batches
    are drawn with the same recipe from a seed of their own."""
    return 1000 + number + 7919 * rank


def local_piece(number: int, world: int, rank: int, mode: str):
    """(global problem, this rank's synth.Inputs, its shard or None).

    batches: the global problem repeats the workload's L batches `world`
    times; rank r owns batches [r L, (r+1) L), drawn with batch_seed(r).
    rows: the global problem is the workload; rank r owns the rows that
    shard.shard_of gives it (whole 128-row scale atoms), as a view of the
    workload's tensors (a rank with no rows gets None)."""
    from block_scaled_precision_04_gb300 import shard as sh
    name, p = synth.WORKLOADS[number]
    if world == 1:
        return p, synth.workload(number), None
    if mode == "batches":
        g = dataclasses.replace(p, L=p.L * world)
        s = sh.shard_of(g.M, g.L, world, rank)
        assert (s.l0, s.l1, s.m0, s.m1) == (rank * p.L, (rank + 1) * p.L, 0, p.M)
        return g, synth.workload(number, seed=batch_seed(number, rank)), s
    if mode != "rows":
        raise ValueError(mode)
    s = sh.shard_of(p.M, p.L, world, rank)
    if s.empty:
        return p, None, s
    full = synth.workload(number)
    C = np.empty(synth.c_shape(p), dtype=np.uint8)  # a stand-in: C views are not kept
    a, b, sfa, sfb, _ = sh.local_views(s, full.A, full.B, full.SFA, full.SFB, C, M=p.M,
                                       a_major=p.a_major, c_major=p.c_major)
    lp = sh.local_problem(p, s)
    return p, synth.Inputs(lp, *(np.ascontiguousarray(x) for x in (a, b, sfa, sfb))), s


def workload_numbers(p: synth.Problem):
    fp4 = p.a_dtype == "e2m1"
    ab = lambda rows: p.L * rows * (p.K // 2 if fp4 else p.K)
    sf = lambda rows: p.L * p.t_k * (-(-rows // 128)) * 512
    c = p.L * p.M * p.N * p.c_itemsize
    flops = 2.0 * p.M * p.N * p.K * p.L
    return {"flops": flops, "bytes": ab(p.M) + ab(p.N) + sf(p.M) + sf(p.N) + c,
            "h2d": ab(p.M) + ab(p.N) + sf(p.M) + sf(p.N), "d2h": c + 4,
            "kind": "fp4" if fp4 else "fp8"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 6800.0, "fallback"


def config_of(number: int, p: synth.Problem, name: str) -> dict:
    return {"workload": name, "M": p.M, "N": p.N, "K": p.K, "L": p.L, "a_dtype": p.a_dtype,
            "b_dtype": p.b_dtype, "sf_vec_size": p.sfv, "sf_dtype": p.sf_dtype,
            "a_major": p.a_major, "b_major": p.b_major,
            "c_dtype": p.c_dtype, "c_major": p.c_major, "seed": 1000 + number,
            "l2": L2_NOTE}


def host_cost_us(launch, torch, dev, n: int = 200):
    """Host time of one launch through the Python binding (argument
    marshalling, the C ABI's checks and the kernel launch), outside the timed
    region: the wall time of a burst of n launches enqueued without waiting,
    per launch.  The class API of the pages is quoted at ~15 us of CPU per
    launch ("GEMM + Amax (SM100)", "Using JAX arrays")."""
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(n):
        launch()
    us = (time.perf_counter() - t0) / n * 1e6
    torch.cuda.synchronize(dev)
    return round(us, 2)


# ------------------------------------------------------------ CPU oracle leg

def oracle_sample(inp, target_s: float, max_rows: int | None = None):
    """Time the oracle (as it stands) on the first r rows of every batch, r
    sized so the run takes about target_s seconds."""
    import oracle
    p = inp.problem
    args = (p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B, inp.SFA, inp.SFB,
            p.sf_dtype)
    # calibrate on enough rows to keep every oracle thread busy (the oracle
    # splits rows over threads), then size the sample; one more resize if the
    # sample ran well short of the target
    kw = {"a_major": p.a_major, "b_major": p.b_major}
    _, _, threads = oracle.gemm(*args, rows=(0, min(p.M, 2)), want_s=False, **kw)
    rows = min(p.M, 4 * max(1, threads))
    if max_rows:
        rows = min(rows, max_rows)
    for attempt in range(3):
        t0 = time.perf_counter()
        _, _, threads = oracle.gemm(*args, rows=(0, rows), want_s=False, **kw)
        t = time.perf_counter() - t0
        want = int(max(2, min(p.M, (target_s / max(t, 1e-3)) * rows)))
        if max_rows:
            want = min(want, max_rows)
        if t >= 0.5 * target_s or want <= rows or attempt == 2:
            break
        rows = want  # measured again on the next pass
    flops = 2.0 * rows * p.N * p.K * p.L
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of every batch (all N, all K): "
                      f"{flops / 1e9:.1f} GFLOP in {t:.1f} s, double precision"}, rows, t


# --------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.split(",") for r in f.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- GPU leg

def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import block_scaled_precision_04_gb300 as bsg

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    name, _ = synth.WORKLOADS[args.workload]
    # the global problem and this rank's piece of it (the whole workload at N = 1)
    g, inp, piece = local_piece(args.workload, world, rank, args.shard)
    if inp is None:
        raise SystemExit(f"rank {rank}: no rows of the workload left for this rank; "
                         f"use fewer GPUs or --shard batches")
    p = inp.problem
    nums = workload_numbers(p)
    global_flops = 2.0 * g.M * g.N * g.K * g.L
    from block_scaled_precision_04_gb300 import shard as sh
    op = bsg.GemmAmax(bsg.make_problem(p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv,
                                       p.c_dtype, p.c_major, sf_dtype=p.sf_dtype,
                                       a_major=p.a_major, b_major=p.b_major),
                      device=local_rank)
    info = op.describe()
    hA, hB, hSFA, hSFB = [torch.from_numpy(np.ascontiguousarray(x)) for x in
                          (inp.A, inp.B, inp.SFA, inp.SFB)]
    A, B, SFA, SFB = [t.to(dev) for t in (hA, hB, hSFA, hSFB)]
    ctype = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[p.c_dtype]
    C = torch.empty(synth.c_shape(p), dtype=ctype, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream

    def launch():
        bsg.check(bsg.bsg_run(op.plan, A.data_ptr(), B.data_ptr(), SFA.data_ptr(),
                              SFB.data_ptr(), C.data_ptr(), amax.data_ptr(),
                              op.workspace.data_ptr(), op.ws_bytes, s), "bsg_run")

    def step():
        # one pass of the path: this rank's launch, then (N > 1) the one
        # exchange, the max of the per-rank Amax over the ranks
        launch()
        if world > 1:
            sh.allreduce_amax(amax)

    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize(dev)
    bsg.check(op.device_status(), "device status (warm-up)")

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        for e0, e1 in evs:
            flush_l2(flush)
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    bsg.check(op.device_status(), "device status")
    times_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_ms = max_over_ranks(sum(times_ms), dist, dev)
    ms = total_ms / args.steps
    # the whole job's work (every rank's piece) over the slowest rank's time
    value = whole_job_tflops(global_flops, args.steps, 1, total_ms)
    host_us = host_cost_us(launch, torch, dev)
    bsg.check(op.device_status(), "device status (host-cost burst)")

    # end to end through the C ABI with host buffers (pinned), copies included.
    # Steps alternate between --e2e-streams streams, each with its own device
    # buffers, workspace and pinned C: a step's input copies then overlap the
    # previous step's kernel and result copy (the link carries both
    # directions at once); every step still copies all of its inputs in and
    # its C and Amax out.
    e2e = None
    if not args.no_e2e:
        pA, pB, pSFA, pSFB = [t.pin_memory() for t in (hA, hB, hSFA, hSFB)]
        n_str = max(1, args.e2e_streams)
        streams = [stream] + [torch.cuda.Stream(dev) for _ in range(n_str - 1)]
        sets = []
        for i, st_i in enumerate(streams):
            if i == 0:
                dv = (A, B, SFA, SFB, C, amax, op.workspace)
            else:
                ws_i = torch.empty(op.ws_bytes, dtype=torch.uint8, device=dev)
                bsg.check(bsg.bsg_workspace_init(op.plan, ws_i.data_ptr(), op.ws_bytes, st_i.cuda_stream),
                          "bsg_workspace_init")
                dv = (torch.empty_like(A), torch.empty_like(B), torch.empty_like(SFA),
                      torch.empty_like(SFB), torch.empty_like(C), torch.zeros_like(amax), ws_i)
            pC = torch.empty(synth.c_shape(p), dtype=ctype).pin_memory()
            pamax = torch.empty(1, dtype=torch.float32).pin_memory()
            bufs = bsg.bsg_device_buffers(*(t.data_ptr() for t in dv[:6]), dv[6].data_ptr(), op.ws_bytes)
            sets.append((st_i, dv, pC, pamax, bufs))
        torch.cuda.synchronize(dev)

        def run_host(k):
            st_i, dv, pC, pamax, bufs = sets[k % n_str]
            bsg.check(bsg.bsg_run_host(
                op.plan, pA.data_ptr(), pB.data_ptr(), pSFA.data_ptr(), pSFB.data_ptr(),
                pC.data_ptr(), pamax.data_ptr(), bufs, st_i.cuda_stream), "bsg_run_host")
            if world > 1:  # the global Amax: reduced on the device, then read back
                with torch.cuda.stream(st_i):
                    sh.allreduce_amax(dv[5])
                    pamax.copy_(dv[5], non_blocking=True)
        for k in range(max(n_str, args.warmup)):
            run_host(k)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st_i in streams[1:]:
            st_i.wait_event(e0)
        for k in range(args.steps):
            run_host(k)
        for st_i in streams[1:]:
            done = torch.cuda.Event()
            done.record(st_i)
            stream.wait_event(done)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
        e2e = {"value": global_flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "streams": n_str, "h2d_bytes_per_step": nums["h2d"],
               "d2h_bytes_per_step": nums["d2h"] + (4 if world > 1 else 0)}

    bf16, hbm, source = peaks()
    peak = bf16 * NOMINAL_RATIO[nums["kind"]]
    achieved = nums["flops"] / (ms / 1e3) / 1e12
    traffic = TRAFFIC.get((kernel_source_hash(), args.workload))
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{source} bf16 {bf16} TFLOP/s x nominal dense "
                               f"{nums['kind']}/bf16 ratio {NOMINAL_RATIO[nums['kind']]:g}",
                "kernel": info["kernel_name"],
                "hbm_gbs_algorithmic": round(nums["bytes"] / (ms / 1e3) / 1e9, 1),
                "hbm_frac_of_" + source: round(nums["bytes"] / (ms / 1e3) / 1e9 / hbm, 4)}
    if nums["kind"] == "fp4":
        # the FP4 rate this part's tensor cores reach: 2x the FP8 peak above
        fp4_reach = bf16 * NOMINAL_RATIO["fp8"] * MEASURED_FP4_OVER_FP8
        roofline["frac_of_measured_fp4_mma_rate"] = round(achieved / fp4_reach, 4)

    line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True,
            "scaling": "strong" if world > 1 and args.shard == "rows" else "weak",
            "vs_baseline": None,
            "dtype": f"{p.a_dtype}x{p.b_dtype} codes, "
                     f"{'e8m0' if p.sf_dtype == 'ue8m0' else p.sf_dtype} scales, fp32 accumulate",
            "data": "synthetic (seeded; see synth)", "config": config_of(args.workload, g, name),
            "roofline": roofline, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": clk.summary(), "wall_s_timed_region": round(wall, 4),
            "host_us_per_launch": host_us,
            "plan": {k: info[k] for k in ("tile_m", "tile_n", "stages", "grid", "smem_bytes",
                                          "num_tiles")},
            "step_ms_min": round(min(times_ms), 5), "step_ms_median": round(statistics.median(times_ms), 5)}
    if world > 1:
        line["config"]["shard"] = {
            "mode": args.shard, "ranks": world,
            "rank0_piece": {"l0": piece.l0, "l1": piece.l1, "m0": piece.m0, "m1": piece.m1},
            "exchange": "all-reduce (int32 max of the fp32 Amax bits) over NCCL, inside every "
                        "timed step"}
    if rank == 0 and not args.no_cpu:
        cb, _, _ = oracle_sample(inp, args.cpu_seconds)
        line["cpu_baseline"] = cb
    elif rank == 0:
        line["cpu_baseline"] = None
    return line


def quant_numbers(rows, cols, in_dtype, out_dtype, sfv, direction="row"):
    x = rows * cols * (4 if in_dtype == "f32" else 2)
    codes = rows * cols // (2 if out_dtype == "e2m1" else 1)
    if direction == "col":
        sf = -(-cols // 128) * -(-(rows // sfv) // 4) * 512
    else:
        sf = -(-rows // 128) * -(-(cols // sfv) // 4) * 512
    return {"bytes": x + codes + sf, "h2d": x, "d2h": codes + sf}


def quant_oracle_sample(X32, out_dtype, sfv, target_s: float, direction="row"):
    """The oracle's quantizer (single thread), timed on the first r rows
    (whole 32-row blocks for the columnwise form), r sized for about
    target_s seconds."""
    import oracle
    step = 32 if direction == "col" else 1
    fn = ((lambda x: oracle.quantize_colwise(x, out_dtype, sfv)) if direction == "col" else
          (lambda x: oracle.quantize(x, out_dtype, sfv)))
    rows = min(X32.shape[1], 64)
    for attempt in range(3):
        t0 = time.perf_counter()
        fn(X32[:, :rows].astype(np.float64))
        t = time.perf_counter() - t0
        want = int(min(X32.shape[1], max(1, (target_s / max(t, 1e-3)) * rows)))
        want = max(step, want // step * step)
        if t >= 0.5 * target_s or want <= rows or attempt == 2:
            break
        rows = want
    return rows, t


def run_quant(args, rank: int, world: int, local_rank: int):
    import torch
    import block_scaled_precision_04_gb300 as bsg

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    name, rows, cols, in_dtype, out_dtype, sfv, direction = QWORKLOADS[args.qworkload]
    gen = synth.real_blocks_colwise if direction == "col" else synth.real_blocks
    X32 = gen(1, rows, cols, seed=1500 + args.qworkload, block=sfv)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[in_dtype]
    hX = torch.from_numpy(X32).to(tdt)
    X = hX.to(dev)
    q = bsg.make_quant_problem(rows, cols, 1, in_dtype, out_dtype, sfv, direction)
    st, (cb, sb) = bsg.bsg_quant_sizes(q)
    bsg.check(st, "bsg_quant_sizes")
    codes = torch.empty(cb, dtype=torch.uint8, device=dev)
    sf = torch.empty(sb, dtype=torch.uint8, device=dev)
    nums = quant_numbers(rows, cols, in_dtype, out_dtype, sfv, direction)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    launch = lambda: bsg.check(bsg.bsg_quantize(q, X.data_ptr(), codes.data_ptr(), sf.data_ptr(), s),
                               "bsg_quantize")
    for _ in range(args.warmup):
        flush_l2(flush)
        launch()
    torch.cuda.synchronize(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        for e0, e1 in evs:
            flush_l2(flush)
            e0.record(stream)
            launch()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    times_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_ms = max_over_ranks(sum(times_ms), dist, dev)
    ms = total_ms / args.steps
    value = world * nums["bytes"] * args.steps / (total_ms / 1e3) / 1e9

    e2e = None
    if not args.no_e2e:
        pX = hX.pin_memory()
        pcodes = torch.empty(cb, dtype=torch.uint8).pin_memory()
        psf = torch.empty(sb, dtype=torch.uint8).pin_memory()

        def run_host():
            X.copy_(pX, non_blocking=True)
            launch()
            pcodes.copy_(codes, non_blocking=True)
            psf.copy_(sf, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            run_host()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            run_host()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
        e2e = {"value": world * nums["bytes"] / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": nums["h2d"],
               "d2h_bytes_per_step": nums["d2h"]}

    _, hbm, source = peaks()
    achieved = nums["bytes"] / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(hbm, 1),
                "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": TRAFFIC_Q.get((kernel_source_hash("quant.cu"), args.qworkload)),
                "peak_source": f"{source} HBM copy bandwidth",
                "kernel": "bsq_quantize_colwise_kernel" if direction == "col" else
                          "bsq_quantize_kernel"}
    line = {"metric": QMETRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": f"{in_dtype} in, {out_dtype} codes + e8m0 scales out"
                     f"{' (columnwise blocks)' if direction == 'col' else ''}",
            "data": "synthetic (seeded; see synth.real_blocks)",
            "config": {"workload": name, "rows": rows, "cols": cols, "L": 1, "in_dtype": in_dtype,
                       "out_dtype": out_dtype, "sf_vec_size": sfv, "direction": direction,
                       "seed": 1500 + args.qworkload, "l2": L2_NOTE},
            "roofline": roofline, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": clk.summary(), "wall_s_timed_region": round(wall, 4),
            "step_ms_min": round(min(times_ms), 5),
            "step_ms_median": round(statistics.median(times_ms), 5)}
    if rank == 0 and not args.no_cpu:
        r, t = quant_oracle_sample(X32 if in_dtype == "f32" else hX.float().numpy(), out_dtype, sfv,
                                   args.cpu_seconds, direction)
        b = quant_numbers(r, cols, in_dtype, out_dtype, sfv, direction)["bytes"]
        line["cpu_baseline"] = {"value": b / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"rows 0..{r - 1} (all columns): {b / 1e6:.1f} MB "
                                          f"in {t:.1f} s, one thread, double precision"}
    elif rank == 0:
        line["cpu_baseline"] = None
    return line


def run_quant_reference(args):
    """The oracle's quantizer, as it stands, on a bounded sample per step."""
    import oracle
    name, rows, cols, in_dtype, out_dtype, sfv, direction = QWORKLOADS[args.qworkload]
    gen = synth.real_blocks_colwise if direction == "col" else synth.real_blocks
    X32 = gen(1, rows, cols, seed=1500 + args.qworkload, block=sfv)
    if in_dtype == "bf16":
        import torch
        X32 = torch.from_numpy(X32).to(torch.bfloat16).float().numpy()
    per_step = max(0.5, args.ref_seconds / max(1, args.steps + args.warmup))
    r, _ = quant_oracle_sample(X32, out_dtype, sfv, per_step, direction)
    Xs = X32[:, :r].astype(np.float64)
    fn = oracle.quantize_colwise if direction == "col" else oracle.quantize
    for _ in range(args.warmup):
        fn(Xs, out_dtype, sfv)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn(Xs, out_dtype, sfv)
    t = time.perf_counter() - t0
    b = quant_numbers(r, cols, in_dtype, out_dtype, sfv, direction)["bytes"]
    value = b * args.steps / t / 1e9
    return {"metric": QMETRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": name, "rows": rows, "cols": cols}, "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"rows 0..{r - 1} per step ({b / 1e6:.1f} MB, double)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_reference(args):
    """The CPU oracle, as it stands, on a bounded sample of the same workload
    per step."""
    name, p = synth.WORKLOADS[args.workload]
    inp = synth.workload(args.workload)
    nums = workload_numbers(p)
    per_step = max(0.5, args.ref_seconds / max(1, args.steps + args.warmup))
    _, rows, _ = oracle_sample(inp, per_step)
    import oracle
    pargs = (p.M, p.N, p.K, p.L, p.a_dtype, p.b_dtype, p.sfv, inp.A, inp.B, inp.SFA, inp.SFB,
             p.sf_dtype)
    kw = {"a_major": p.a_major, "b_major": p.b_major}
    for _ in range(args.warmup):
        oracle.gemm(*pargs, rows=(0, rows), want_s=False, **kw)
    t0 = time.perf_counter()
    threads = 0
    for _ in range(args.steps):
        _, _, threads = oracle.gemm(*pargs, rows=(0, rows), want_s=False, **kw)
    t = time.perf_counter() - t0
    flops = 2.0 * rows * p.N * p.K * p.L
    value = flops * args.steps / t / 1e12
    sample = f"rows 0..{rows - 1} of every batch per step ({flops / 1e9:.1f} GFLOP, double)"
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": config_of(args.workload, p, name), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0, "workload_flops_per_full_step": nums["flops"]}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=None,
                    help="GPUs (one process each); unset: WORLD_SIZE, else 1")
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--op", choices=["gemm", "quantize"], default="gemm")
    ap.add_argument("--shard", choices=["batches", "rows"], default="batches",
                    help="N > 1: batches (each rank L batches of its own, weak scaling) or "
                         "rows (the workload split in 128-row atoms, strong scaling)")
    ap.add_argument("--qworkload", type=int, default=1, choices=sorted(QWORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams the end-to-end GEMM steps alternate between (3: the host "
                         "link carries both directions; more streams measured no faster)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least three warm-up steps

    if "WORLD_SIZE" not in os.environ and (args.gpus or 1) > 1:
        # one process per GPU: run this command under torch.distributed.run
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        argv = sys.argv[1:] if argv is None else list(argv)
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               "--master-port", str(port), os.path.abspath(__file__), *argv]
        return subprocess.call(cmd)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus is not None and args.gpus != world:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
        return 2

    if args.impl == "reference":
        if rank == 0:
            ref = run_quant_reference(args) if args.op == "quantize" else run_reference(args)
            print(json.dumps(ref), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = (run_quant if args.op == "quantize" else run_ours)(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
