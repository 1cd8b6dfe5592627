"""Benchmark of the dense GEMM C = A·Bᵀ (fp16 in, fp32 accumulate and out).

One step = one call of each shape of the workload, each call timed alone with
CUDA events on the launching stream, an L2 flush (a 256 MiB write) between
calls, nothing overlapping ("SASS-Level Kernel Generation for Blackwell",
section "How we measured": every call runs alone). Inputs are seeded
synthetic uniform[-1, 1] fp16 matrices, resident in HBM before timing starts.

Default workload: the square and near-square sweep (1536³, 2048³, 4096³,
3072×1280×2048, 4096×4096×1024, 8192×2048×4096). Other workloads: c1
(1024³), splitk (1024×1024×65536), streamk (2048×2048×16384), large (8192³,
16384³), all.

Prints one JSON line (rank 0). `value` = Σ 2·M·N·K over the step's calls ÷
Σ their GPU times, in TFLOP/s, over all ranks (replicas for N > 1).

`--impl reference` times the CPU oracle (the plain fp64 triple loop) on the
host cores, on a bounded row sample of the same shapes, in the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

from dense_fp16_gemm_02_gb300.clocks import ClockSampler

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("µs/call and TFLOP/s per shape (1 GB300) + fraction of dense fp16 tensor peak")
# Operand and C element types: the pages' product (fp16 -> fp32) and the
# adjacent variants of the same kernels.
TYPES = {"f16f32": ("f16", "f32"), "bf16f32": ("bf16", "f32"), "f16f16": ("f16", "f16"),
         "bf16bf16": ("bf16", "bf16")}

WORKLOADS = {
    "c1": [(1024, 1024, 1024)],
    "sweep": [(1536, 1536, 1536), (2048, 2048, 2048), (4096, 4096, 4096), (3072, 1280, 2048),
              (4096, 4096, 1024), (8192, 2048, 4096)],
    "splitk": [(1024, 1024, 65536)],
    "streamk": [(2048, 2048, 16384)],
    "large": [(8192, 8192, 8192), (16384, 16384, 16384)],
}
WORKLOADS["all"] = (WORKLOADS["c1"] + WORKLOADS["sweep"] + WORKLOADS["large"]
                    + WORKLOADS["streamk"] + WORKLOADS["splitk"])
MODE_NAMES = ["data-parallel", "split-K", "stream-K", "data-parallel + stream-K tail"]
FLUSH_BYTES = 256 << 20  # > the 129 MB L2
GATE_CYCLES = 400_000    # ≈ 0.2 ms of GPU spin ahead of each timed call
FALLBACK_TFLOPS = 1900.0
FALLBACK_TFLOPS_SUSTAINED = 1700.0
FALLBACK_HBM_GBS = 6800.0


def shape_name(s):
    return "x".join(str(v) for v in s)


def peaks(power_capped: bool = False):
    """(tensor TFLOP/s, HBM GB/s, source). The tensor figure is the measured
    cuBLAS bf16 rate (fp16 runs at the same nominal rate): the burst figure,
    or the sustained one when the timed region ran under the power cap (a
    long run of back-to-back large GEMMs), since that is the regime the
    sustained figure was measured in."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if power_capped and "bf16_tflops_sustained" in d:
            return (float(d["bf16_tflops_sustained"]), float(d["hbm_gbs"]),
                    "measured: bf16 cuBLAS sustained (timed region under sw_power_cap)")
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured: bf16 cuBLAS burst"
    except (OSError, KeyError, ValueError):
        if power_capped:
            return FALLBACK_TFLOPS_SUSTAINED, FALLBACK_HBM_GBS, "fallback: sustained"
        return FALLBACK_TFLOPS, FALLBACK_HBM_GBS, "fallback: burst"


KERNEL_SOURCES = ["wgemm_kernel.cuh", "wgemm_plan.h", "wgemm_configs.h", "inst_single.cu",
                  "inst_pair.cu", "inst_pair2.cu", "inst_multicast.cu", "inst_clc.cu",
                  "inst_out16_a.cu", "inst_out16_b.cu", "inst_fused.cu", "inst_rowmc.cu", "sm103/ptx.cuh",
                  "sm103/umma_desc.h"]


def _code_only(text: str) -> str:
    """C/C++ source without comments and whitespace (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':  # string literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c.isspace():
            i += 1
        else:
            out.append(c)
            i += 1
    return "".join(out)


def kernel_source_digest() -> str:
    """Digest of the code (comments and whitespace removed) of the files that
    define the GEMM kernels (not the host code)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp16_gemm_02_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(config_name: str, shape):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources for this configuration and shape."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rows = json.load(f)
    except (OSError, ValueError):
        return None
    digest = kernel_source_digest()
    for r in rows:
        if (r.get("kernel_src") == digest and r.get("config") == config_name
                and r.get("shape") == shape_name(shape)):
            return r.get("dram_bytes")
    return None


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity with
    one process). Every rank's timed region is bracketed by barriers, so the
    slowest rank's time is the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_value(flops_per_rank_step: float, world: int, step_ms: float) -> float:
    """Whole-job throughput in TFLOP/s: every rank's flops over the slowest time."""
    return world * flops_per_rank_step / (step_ms * 1e-3) / 1e12


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


_B_CACHE = {}
_A_CACHE = {}
_CAL_CACHE = {}


def oracle_sample_rate(shapes, seconds_total: float, nthreads: int = 0, ab: str = "f16"):
    """Times the CPU oracle on a row sample of every shape, about
    `seconds_total` of oracle work in all (a shape that finishes in full hands
    its unused share to the larger ones). A call's cost is a fixed part (the
    oracle decodes all of B first) plus a cost per row of A; the fixed part
    is calibrated once per shape, and each shape's full call is estimated as
    fixed + (sample time - fixed) · M / rows. Returns (TFLOP/s over the
    estimated full calls, threads, description, seconds of oracle work)."""
    import oracle
    from dense_fp16_gemm_02_gb300 import inputs
    total_flops, total_t, work, desc = 0.0, 0.0, 0.0, []
    threads = nthreads or oracle.hardware_threads()
    order = sorted(range(len(shapes)), key=lambda i: shapes[i][0] * shapes[i][1] * shapes[i][2])
    left = seconds_total
    for n_done, i in enumerate(order):
        M, N, K = shapes[i]
        budget = left / (len(order) - n_done)
        if (N, K, ab) not in _B_CACHE:
            _B_CACHE[(N, K, ab)] = inputs.matrix(N, K, 1000, 1, dtype=ab)
        B = _B_CACHE[(N, K, ab)]
        # Calibrate (once per shape and thread count) at one and at four rows
        # per thread. Then size the sample to the budget.
        key = (M, N, K, ab, threads)
        if key not in _CAL_CACHE:
            cal = []
            for r in sorted({min(M, threads), min(M, 4 * threads)}):
                A = inputs.matrix(r, K, 1000, 0, dtype=ab)
                t0 = time.perf_counter()
                oracle.gemm_f64(A, B, nthreads=threads)
                cal.append((r, time.perf_counter() - t0))
            if len(cal) == 2:
                (r1, t1), (r2, t2) = cal
                per_row = max((t2 - t1) / (r2 - r1), t2 / r2 * 0.05, 1e-7)
                fixed = max(t1 - per_row * r1, 0.0)
            else:
                per_row, fixed = max(cal[0][1], 1e-4) / cal[0][0], 0.0
            _CAL_CACHE[key] = (per_row, fixed)
        per_row, fixed = _CAL_CACHE[key]
        rows = min(M, threads)
        rows = int(min(M, max(rows, (budget - fixed) / per_row)))
        if rows > threads:
            rows -= rows % threads
        akey = (M, K, ab)
        if akey not in _A_CACHE or _A_CACHE[akey].shape[0] < rows:
            _A_CACHE[akey] = inputs.matrix(rows, K, 1000, 0, dtype=ab)
        A = _A_CACHE[akey][:rows]
        t0 = time.perf_counter()
        oracle.gemm_f64(A, B, nthreads=threads)
        dt = time.perf_counter() - t0
        left -= dt
        work += dt
        full = dt if rows == M else fixed + max(dt - fixed, 0.0) * M / rows
        total_flops += 2.0 * M * N * K
        total_t += full
        desc.append(f"{rows} of {M} rows of {shape_name((M, N, K))}")
    return total_flops / total_t / 1e12, threads, "; ".join(desc), work


def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    shapes = WORKLOADS[args.workload]
    # About 150 s of oracle work over the whole run, however many steps.
    budget = max(0.02 * len(shapes), min(60.0, 150.0 / max(1, args.steps + args.warmup)))
    ab = TYPES[args.types][0]
    for _ in range(args.warmup):
        oracle_sample_rate(shapes, budget / 4, ab=ab)
    vals, last = [], None
    for _ in range(args.steps):
        last = oracle_sample_rate(shapes, budget, ab=ab)
        vals.append(last[0])
    value = statistics.median(vals)
    tflop_per_step = sum(2.0 * M * N * K for (M, N, K) in shapes) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tflop_per_step / value * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload + ": " + ", ".join(shape_name(s) for s in shapes),
                   "types": args.types,
                   "oracle": "plain fp64 triple loop in C (oracle/wgemm_oracle.c)",
                   "sample": ("row sample per shape; each full call estimated as the "
                              "calibrated fixed cost (decoding B) plus the sample's "
                              "per-row time times M")},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last[1], "kind": "oracle",
                         "sample": last[2]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch

    from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    build.build()
    wgemm.load()
    shapes = WORKLOADS[args.workload]
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    ab, c = TYPES[args.types]
    ab_type = wgemm.WGEMM_F16 if ab == "f16" else wgemm.WGEMM_BF16
    c_type = {"f32": wgemm.WGEMM_F32, "f16": wgemm.WGEMM_F16, "bf16": wgemm.WGEMM_BF16}[c]
    c_torch = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[c]
    c_bytes = 4 if c == "f32" else 2

    def as_tensor(x):  # fp16 arrays, or bf16 bit patterns (uint16)
        t = torch.from_numpy(x if ab == "f16" else x.view(np.int16))
        return t if ab == "f16" else t.view(torch.bfloat16)

    # Inputs: generated on the host once, uploaded before timing.
    data = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = inputs.gemm_operands(M, N, K, seed=1000 + i, kind=args.values, dtype=ab)
        dA, dB = as_tensor(A).to(dev), as_tensor(B).to(dev)
        C = torch.zeros((M, N), dtype=c_torch, device=dev)
        data.append((A, B, dA, dB, C))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    names = wgemm.config_names()

    fused = args.epilogue == "fused"
    biases = [torch.from_numpy(inputs.matrix(1, N, 2000 + i, 6, "uniform").astype(np.float32)
                               .ravel()).to(dev) for i, (M, N, K) in enumerate(shapes)]

    def call(i):
        (M, N, K) = shapes[i]
        _, _, dA, dB, C = data[i]
        if fused:  # D = A·Bᵀ + D + bias: the previous result read back in place
            rc = wgemm.wgemm_gemm_ex(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), C.data_ptr(),
                                     biases[i].data_ptr(), 1.0, 1.0, ab_type, c_type, M, N, K,
                                     K, K, N, N, h)
        elif ab_type == wgemm.WGEMM_F16 and c_type == wgemm.WGEMM_F32:
            rc = wgemm.wgemm_f16f32(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K, N,
                                    h)
        else:
            rc = wgemm.wgemm_gemm(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), ab_type, c_type, M,
                                  N, K, K, K, N, h)
        if rc != 0:
            raise RuntimeError(f"wgemm call failed: {rc}")

    def one_step(events):
        for i in range(len(shapes)):
            flush.fill_(float(i))  # evict L2
            # Keep the GPU busy while the host enqueues the start event and the
            # call, so the event pair brackets the kernel, not host latency.
            torch.cuda._sleep(GATE_CYCLES)
            e0, e1 = events[i]
            e0.record(stream)
            call(i)
            e1.record(stream)

    mk = lambda: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in shapes]
    for _ in range(args.warmup):
        one_step(mk())
    rc = wgemm.wgemm_check(h)
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {wgemm.wgemm_last_device_error()}")

    per_step_events = [mk() for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        clocks.mark_start()
        t_wall = time.perf_counter()
        for s in range(args.steps):
            one_step(per_step_events[s])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clocks.mark_stop()
    if world > 1:
        dist.barrier()
    rc = wgemm.wgemm_check(h)
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {wgemm.wgemm_last_device_error()}")
    gpu_launches = args.steps * len(shapes)

    times = np.array([[e0.elapsed_time(e1) for (e0, e1) in ev] for ev in per_step_events])  # ms
    step_ms = float(np.median(times.sum(axis=1)))
    flops = np.array([2.0 * M * N * K for (M, N, K) in shapes])
    step_ms = max_over_ranks([step_ms], dev)[0]
    value = job_value(float(flops.sum()), world, step_ms)
    clk = clocks.summary()
    peak_tflops, peak_hbm, peak_src = peaks("sw_power_cap" in clk["reasons"])

    # Per-shape report, and the configuration each call ran.
    per_shape = []
    by_config = {}
    for i, (M, N, K) in enumerate(shapes):
        us = times[:, i] * 1e3
        # The fused bench call is in place with beta = 1: with fp32 D it may
        # also take the reduce-add kernels (fused kind 2).
        fused_kind = 0 if args.epilogue != "fused" else (2 if c_type == wgemm.WGEMM_F32 else 1)
        cfg, mode, splits = wgemm.wgemm_select(M, N, K, c_type=c_type, fused=fused_kind)
        med = float(np.median(us))
        tf = flops[i] / (med * 1e-6) / 1e12
        c_rw = (2 if args.epilogue == "fused" else 1) * c_bytes * M * N  # C written (and read)
        bytes_min = 2.0 * (M * K + N * K) + c_rw
        per_shape.append({
            "shape": shape_name((M, N, K)), "us_median": round(med, 3),
            "us_min": round(float(us.min()), 3), "us_max": round(float(us.max()), 3),
            "tflops": round(tf, 1), "tensor_frac": round(tf / peak_tflops, 4),
            "hbm_gbs": round(bytes_min / (med * 1e-6) / 1e9, 1),
            "hbm_frac": round(bytes_min / (med * 1e-6) / 1e9 / peak_hbm, 4),
            "config": names[cfg], "mode": MODE_NAMES[mode],
            "splits": splits})
        agg = by_config.setdefault(names[cfg], {"flops": 0.0, "ms": 0.0, "launches": 0,
                                                "shape": (M, N, K), "shape_ms": 0.0})
        agg["flops"] += flops[i] * args.steps
        agg["ms"] += float(times[:, i].sum())
        agg["launches"] += args.steps
        if float(times[:, i].sum()) > agg["shape_ms"]:
            agg["shape"], agg["shape_ms"] = (M, N, K), float(times[:, i].sum())
    dom_name, dom = max(by_config.items(), key=lambda kv: kv[1]["ms"])
    achieved = dom["flops"] / (dom["ms"] * 1e-3) / 1e12

    # End to end through the public API with host buffers: every step copies
    # every shape's A and B from pinned host memory to the device, calls the
    # library, and copies C back, all inside the timed region. The copies run
    # on their own streams, pipelined across the step's shapes as a user
    # would run them: shape i's upload overlaps shape i-1's call and shape
    # i-2's download (the two copy directions use separate copy engines).
    pinned = []
    for (A, B, _, _, C) in data:
        hA = as_tensor(A).pin_memory()
        hB = as_tensor(B).pin_memory()
        hC = torch.empty(C.shape, dtype=c_torch).pin_memory()
        hCin = torch.zeros(C.shape, dtype=c_torch).pin_memory() if fused else None
        pinned.append((hA, hB, hC, hCin))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms = []
    for s in range(e2e_steps + 1):
        flush.fill_(0.0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        stream.wait_event(e0)
        s_out.wait_event(e0)
        for i, (M, N, K) in enumerate(shapes):
            hA, hB, hC, hCin = pinned[i]
            _, _, dA, dB, C = data[i]
            uploaded, computed = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                if hCin is not None:  # the fused epilogue's Cin is an input too
                    C.copy_(hCin, non_blocking=True)
                uploaded.record(s_in)
            stream.wait_event(uploaded)
            call(i)
            computed.record(stream)
            s_out.wait_event(computed)
            with torch.cuda.stream(s_out):
                hC.copy_(C, non_blocking=True)
        e1.record(s_out)
        e1.synchronize()
        if s > 0:  # the first pass warms the copy engines
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_step_ms = max_over_ranks([statistics.median(e2e_ms)], dev)[0]
    h2d = sum(2 * (M * K + N * K) + (c_bytes * M * N if fused else 0) for (M, N, K) in shapes)
    d2h = sum(c_bytes * M * N for (M, N, K) in shapes)

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            rate, cores, sample, secs = oracle_sample_rate(shapes, args.cpu_seconds, ab=ab)
            cpu = {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                   "sample": (f"{sample} ({secs:.1f} s of oracle work; rows not timed "
                              "are estimated from the sample's per-row time plus the "
                              "calibrated fixed cost of decoding B)")}
        line = {
            "metric": METRIC, "value": round(float(value), 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ab, "data": "synthetic",
            "config": {
                "workload": args.workload + ": " + ", ".join(shape_name(s) for s in shapes),
                "inputs": (f"uniform[-1,1] rounded to {ab}" if args.values == "uniform" else
                           "integers in {-2..2}") + ", seeded SplitMix64, resident in HBM",
                "accumulate": "f32", "output": c,
                "epilogue": ("D = A·Bᵀ + D + bias (fused; C read back in place)"
                             if args.epilogue == "fused" else "C = A·Bᵀ"),
                "l2": "flushed between calls (256 MiB write), each call timed alone",
                "timing": ("CUDA events on the launching stream around each call; a GPU-side "
                       "spin ahead of the start event hides host enqueue latency"),
                "e2e": ("every step: A and B uploaded from pinned host memory, the call, C "
                        "downloaded; uploads and downloads on two copy streams, pipelined "
                        "across the step's shapes; timed from the first upload to the last "
                        "download"),
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "shapes": per_shape,
            "roofline": {
                "bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 1),
                "peak": peak_tflops, "unit": "TFLOP/s", "frac": round(achieved / peak_tflops, 4),
                "peak_source": f"{peak_src} x fp16/bf16 nominal ratio 1",
                "traffic": committed_traffic(dom_name, dom["shape"]),
                "traffic_shape": shape_name(dom["shape"]),
            },
            "cpu_baseline": cpu,
            "e2e": {"value": round(job_value(float(flops.sum()), world, e2e_step_ms), 2),
                    "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": gpu_launches,
            "clocks": clk,
            "wall_s_timed": round(t_wall, 3),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    # 200 steps of the sweep take about a third of a second: with clocks
    # sampled every 50 ms, several samples fall inside the timed region.
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="sweep")
    ap.add_argument("--shape", metavar="MxNxK",
                    help="time this one shape instead of a named workload")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="oracle time budget of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--types", choices=sorted(TYPES), default="f16f32",
                    help="operand and C types (the measured product is f16f32)")
    ap.add_argument("--values", choices=["uniform", "int"], default="uniform",
                    help="operand values: uniform[-1,1] (the metric) or the integer copy")
    ap.add_argument("--epilogue", choices=["plain", "fused"], default="plain",
                    help="fused: D = A·Bᵀ + D + bias through the alpha/beta/bias epilogue")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.shape:
        dims = tuple(int(v) for v in args.shape.lower().split("x"))
        if len(dims) != 3 or min(dims) <= 0:
            ap.error("--shape wants MxNxK")
        WORKLOADS["shape"] = [dims]
        args.workload = "shape"
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
