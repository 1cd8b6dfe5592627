"""Benchmark of the dense GEMM C = A·Bᵀ (fp16 in, fp32 accumulate and out).

One step = a pass over every shape of the workload. Each shape is called
several times per step (more often for small shapes, as the pages time
400 calls of a small shape and a dozen of the largest), every call timed
alone with CUDA events on the launching stream, after an L2 flush (a
256 MiB write) and a GPU-side gate, nothing overlapping ("SASS-Level Kernel
Generation for Blackwell", section "How we measured": every call runs
alone). Inputs are seeded synthetic uniform[-1, 1] fp16 matrices, resident
in HBM before timing starts.

Default workload: all eleven shapes of the pages' table ("The numbers"):
1024³, the square and near-square sweep (1536³, 2048³, 4096³,
3072×1280×2048, 4096×4096×1024, 8192×2048×4096), 8192³, 16384³, the stream-K
case 2048×2048×16384 and the split-K case 1024×1024×65536. Named subsets:
c1, sweep, large, streamk, splitk.

After the timed steps, a second pass records every call's GPU kernel time
with CUPTI (the pages' measure: kernel time, median over the calls), once
with the L2 flushed before each call and once with a warm L2 and a device
synchronisation after each call (the pages' protocol).

Prints one JSON line. `value` = Σ 2·M·N·K over a step's calls ÷ the step's
summed GPU event time, in TFLOP/s. One GPU only: the library's cluster
kernels multicast TMA loads within a cluster, which stays a one-GPU feature.

`--impl reference` times the CPU oracle (the plain fp64 triple loop) on the
host cores, on a bounded row sample of the same shapes, in the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
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
MODE_NAMES = ["data-parallel", "split-K", "stream-K", "data-parallel + stream-K tail",
              "stream-K, zeroing first"]


def calls_per_step(M: int, N: int, K: int) -> int:
    """Calls of a shape in one step: the pages time 400 calls of the small
    shapes, 200 of the ~75 µs ones, 40 at 8192³ and 12 at 16384³ ("How we
    measured"); a step holds three times a twentieth of that (so 20 steps
    hold three times the pages' count), which keeps the timed region several
    seconds long, for a clock record with many samples under load."""
    flops = 2.0 * M * N * K
    if flops >= 4e12:
        return 2
    if flops >= 5e11:
        return 6
    if flops >= 1e11:
        return 30
    return 60


FLUSH_BYTES = 256 << 20  # > the 129 MB L2
GATE_CYCLES = 400_000    # ≈ 0.2 ms of GPU spin ahead of each timed call
FALLBACK_TFLOPS = 1900.0
FALLBACK_TFLOPS_SUSTAINED = 1700.0
FALLBACK_HBM_GBS = 6800.0


def shape_name(s):
    return "x".join(str(v) for v in s)


def peaks():
    """(tensor TFLOP/s burst, tensor TFLOP/s sustained, HBM GB/s, source). The
    tensor figures are the measured cuBLAS bf16 rates (fp16 runs at the same
    nominal rate). Every call is timed alone, so the burst figure is the
    denominator; the sustained one (a seconds-long loop under the power cap)
    is reported beside it."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return (float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                float(d["hbm_gbs"]), "measured: bf16 cuBLAS burst")
    except (OSError, KeyError, ValueError):
        return FALLBACK_TFLOPS, FALLBACK_TFLOPS_SUSTAINED, FALLBACK_HBM_GBS, "fallback: burst"


def pipe_ceiling():
    """(TFLOP/s, description) of the tensor pipe on its own: the largest rate
    of the tcgen05.mma microbenchmark (dense_fp16_gemm_02_gb300/peak.py),
    back-to-back MMAs on operands resident in shared memory, all SMs, from
    the committed profiles/tensor_pipe_ceiling.json; None if absent."""
    path = os.path.join(ROOT, "profiles", "tensor_pipe_ceiling.json")
    try:
        with open(path) as f:
            d = json.load(f)
        best = max(d["shapes"], key=lambda r: r["tflops"])
        return float(best["tflops"]), f"tcgen05.mma microbenchmark, {best['mma']} (the largest)"
    except (OSError, KeyError, ValueError):
        return None, None


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


def job_value(flops_per_step: float, step_ms: float) -> float:
    """Throughput in TFLOP/s: a step's flops over the step's time."""
    return flops_per_step / (step_ms * 1e-3) / 1e12


def workload_config(args, shapes):
    """The workload description, the same for both arms."""
    ab, c = TYPES[args.types]
    return {
        "workload": args.workload + ": " + ", ".join(shape_name(s) for s in shapes),
        "inputs": (f"uniform[-1,1] rounded to {ab}" if args.values == "uniform" else
                   "integers in {-2..2}") + ", seeded SplitMix64",
        "accumulate": "f32", "output": c,
        "epilogue": ("D = A·Bᵀ + D + bias (fused; C read back in place)"
                     if args.epilogue == "fused" else "C = A·Bᵀ"),
        "parallelism": "single GPU",
    }


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


def single_gpu_only(args) -> str | None:
    """The reason this run cannot go ahead, or None. The bench runs one GPU:
    its cluster kernels multicast TMA loads within a cluster, which is kept to
    one-GPU runs, and the path has no exchange step to measure."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != 1 or world != 1:
        return (f"one GPU only (asked for --gpus {args.gpus}, WORLD_SIZE {world}): the GEMM "
                "runs on one GPU and its cluster kernels multicast TMA loads within a cluster")
    return None


def run_reference(args):
    shapes = WORKLOADS[args.workload]
    # About 100 s of sampled oracle work over the whole run, however many
    # steps (each call also decodes all of B, which 16384³ makes 2 GB of fp64).
    budget = max(0.02 * len(shapes), min(60.0, 100.0 / max(1, args.steps + args.warmup)))
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
        "config": workload_config(args, shapes),
        "timing": {"oracle": "plain fp64 triple loop in C (oracle/wgemm_oracle.c), host cores",
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


def _median(xs):
    return float(statistics.median(xs)) if xs else None


def run_ours(args):
    import numpy as np
    import torch

    from dense_fp16_gemm_02_gb300 import build, inputs, ktime, wgemm

    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    build.build()
    lib = wgemm.load()
    if args.no_cooperative:  # for Nsight Compute, which cannot profile cooperative launches
        lib.wgemm_debug_set_cooperative(0)
    shapes = WORKLOADS[args.workload]
    reps = [args.calls or calls_per_step(*s) for s in shapes]
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

    forced = wgemm.config_id(args.config) if args.config else None

    def call(i):
        (M, N, K) = shapes[i]
        _, _, dA, dB, C = data[i]
        if forced is not None:  # a forced configuration and K decomposition
            rc = wgemm.wgemm_gemm_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), ab_type,
                                         c_type, M, N, K, K, K, N, forced, args.mode,
                                         args.splits, h)
        elif fused:  # D = A·Bᵀ + D + bias: the previous result read back in place
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

    # The calls of one step, in order: every shape `reps` times in a row.
    order = [i for i in range(len(shapes)) for _ in range(reps[i])]

    def one_step(events):
        for j, i in enumerate(order):
            flush.fill_(float(j))  # evict L2
            # Keep the GPU busy while the host enqueues the start event and the
            # call, so the event pair brackets the kernel, not host latency.
            torch.cuda._sleep(GATE_CYCLES)
            e0, e1 = events[j]
            e0.record(stream)
            call(i)
            e1.record(stream)

    mk = lambda: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in order]
    for _ in range(args.warmup):
        one_step(mk())
    rc = wgemm.wgemm_check(h)
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {wgemm.wgemm_last_device_error()}")

    per_step_events = [mk() for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(0) as clocks:
        clocks.mark_start()
        t_wall = time.perf_counter()
        for s in range(args.steps):
            one_step(per_step_events[s])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clocks.mark_stop()
    rc = wgemm.wgemm_check(h)
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {wgemm.wgemm_last_device_error()}")
    gpu_launches = args.steps * len(order)  # one GEMM kernel per call (K > 0)

    times = np.array([[e0.elapsed_time(e1) for (e0, e1) in ev] for ev in per_step_events])  # ms
    step_ms = float(np.median(times.sum(axis=1)))
    flops = np.array([2.0 * M * N * K for (M, N, K) in shapes])
    flops_per_step = float(sum(flops[i] for i in order))
    value = job_value(flops_per_step, step_ms)
    clk = clocks.summary()
    peak_tflops, peak_sustained, peak_hbm, peak_src = peaks()
    ceiling, ceiling_src = pipe_ceiling()

    # Kernel-only times from CUPTI, outside the timed region: per shape, calls
    # after an L2 flush and the gate (as timed above), then the pages'
    # protocol: a warm L2, each call followed by a device synchronisation, one
    # untimed call first. Shapes go smallest first, so that the largest (which
    # run into the power cap back to back) do not lower the clock of the rest.
    ktimes, ktime_note = None, None
    if not args.no_kernel_time:
        try:
            rec = ktime.KernelTimes()
            n_k = max(5, min(20, args.steps))
            kinds = []
            torch.cuda.synchronize()
            rec.start()
            by_size = sorted(range(len(shapes)), key=lambda i: flops[i])
            for i in by_size:
                for r in range(n_k):
                    flush.fill_(float(r))
                    torch.cuda._sleep(GATE_CYCLES)
                    call(i)
                    kinds.append((i, "flushed"))
                torch.cuda.synchronize()
                for r in range(n_k + 1):
                    call(i)
                    torch.cuda.synchronize()
                    kinds.append((i, "warm" if r > 0 else "skip"))
            rec.stop()
            recs = [r for r in rec.records() if "wgemm_" in r[0]]
            if len(recs) != len(kinds):
                raise ktime.KernelTimesUnavailable(
                    f"{len(recs)} GEMM kernel records for {len(kinds)} calls "
                    f"({rec.dropped()} dropped)")
            ktimes = {}
            for (i, kind), (_, t0, t1, _) in zip(kinds, recs):
                ktimes.setdefault((i, kind), []).append((t1 - t0) * 1e-3)  # µs
            ktime_note = (f"CUPTI CONCURRENT_KERNEL records; {n_k} calls per shape after an L2 "
                          f"flush, and {n_k} with a warm L2 and a device synchronisation after "
                          "each call (one untimed call first)")
        except ktime.KernelTimesUnavailable as e:
            ktimes, ktime_note = None, f"unavailable: {e}"
    rc = wgemm.wgemm_check(h)
    if rc != 0:
        raise RuntimeError(f"device status {rc}: {wgemm.wgemm_last_device_error()}")

    # Per-shape report, and the configuration each call ran.
    per_shape = []
    by_config = {}
    for i, (M, N, K) in enumerate(shapes):
        cols = [j for j, x in enumerate(order) if x == i]
        us = times[:, cols].ravel() * 1e3
        # The fused bench call is in place with beta = 1: with fp32 D it may
        # also take the reduce-add kernels (fused kind 2).
        fused_kind = 0 if args.epilogue != "fused" else (2 if c_type == wgemm.WGEMM_F32 else 1)
        cfg, mode, splits = wgemm.wgemm_select(M, N, K, c_type=c_type, fused=fused_kind)
        if forced is not None:
            cfg = forced
            mode = args.mode if args.mode >= 0 else mode
            splits = args.splits
        med = float(np.median(us))
        tf = flops[i] / (med * 1e-6) / 1e12
        c_rw = (2 if args.epilogue == "fused" else 1) * c_bytes * M * N  # C written (and read)
        bytes_min = 2.0 * (M * K + N * K) + c_rw
        row = {
            "shape": shape_name((M, N, K)), "calls": int(us.size), "us_median": round(med, 3),
            "us_min": round(float(us.min()), 3), "us_max": round(float(us.max()), 3),
            "tflops": round(tf, 1), "tensor_frac": round(tf / peak_tflops, 4),
            "pipe_frac": round(tf / ceiling, 4) if ceiling else None,
            "hbm_gbs": round(bytes_min / (med * 1e-6) / 1e9, 1),
            "hbm_frac": round(bytes_min / (med * 1e-6) / 1e9 / peak_hbm, 4),
            "config": names[cfg], "mode": MODE_NAMES[mode], "splits": splits}
        if ktimes is not None:
            kf, kw = ktimes.get((i, "flushed"), []), ktimes.get((i, "warm"), [])
            row.update({
                "us_kernel_median": round(_median(kf), 3), "us_kernel_min": round(min(kf), 3),
                "us_kernel_max": round(max(kf), 3),
                "tflops_kernel": round(flops[i] / (_median(kf) * 1e-6) / 1e12, 1),
                "us_kernel_warm_median": round(_median(kw), 3),
                "tflops_kernel_warm": round(flops[i] / (_median(kw) * 1e-6) / 1e12, 1)})
        per_shape.append(row)
        agg = by_config.setdefault(names[cfg], {"flops": 0.0, "ms": 0.0, "launches": 0,
                                                "shape": (M, N, K), "shape_ms": 0.0,
                                                "kernel_us": 0.0, "kernel_flops": 0.0})
        shape_ms = float(times[:, cols].sum())
        agg["flops"] += flops[i] * us.size
        agg["ms"] += shape_ms
        agg["launches"] += int(us.size)
        if ktimes is not None:
            agg["kernel_us"] += _median(ktimes[(i, "flushed")])
            agg["kernel_flops"] += flops[i]
        if shape_ms > agg["shape_ms"]:
            agg["shape"], agg["shape_ms"] = (M, N, K), shape_ms
    dom_name, dom = max(by_config.items(), key=lambda kv: kv[1]["ms"])
    achieved = dom["flops"] / (dom["ms"] * 1e-3) / 1e12

    # End to end through the public API with host buffers: every step copies
    # every shape's A and B from pinned host memory to the device, computes,
    # and copies C back, all inside the timed region. For fp16 → fp32 C the
    # library's host-buffer call does it (wgemm_f16f32_host: A up in row
    # panels and B in blocks of its rows, each GEMM piece starting as its
    # operands land, C down piece by piece), each shape on a stream of its
    # own, as independent calls: one shape's copies overlap another's GEMMs.
    # A call joins its caller's stream to its downloads, so a stream shared by
    # two shapes would hold the second one's uploads behind the first one's
    # downloads. The other element types and the fused
    # epilogue copy on two streams of their own around the device call,
    # pipelined across the step's shapes: shape i's upload overlaps shape
    # i-1's call and shape i-2's download.
    host_entry = ab == "f16" and c == "f32" and not fused and forced is None
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
    if host_entry:
        # The host call's device layout: K rounded up to 8, N up to 4; the
        # bench's device buffers are dense, so every shape must have both.
        assert all(K % 8 == 0 and N % 4 == 0 for (M, N, K) in shapes)
        call_streams = [torch.cuda.Stream(device=dev) for _ in shapes]
    for s in range(e2e_steps + 1 if host_entry else 0):
        flush.fill_(0.0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for cs in call_streams:
            cs.wait_event(e0)
        for i, (M, N, K) in enumerate(shapes):
            hA, hB, hC, _ = pinned[i]
            _, _, dA, dB, C = data[i]
            cs = call_streams[i]
            rc = wgemm.wgemm_f16f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N, K, K,
                                         K, N, dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                                         cs.cuda_stream)
            if rc != 0:
                raise RuntimeError(f"wgemm_f16f32_host failed: {wgemm.status_string(rc)}")
        for cs in call_streams:
            stream.wait_stream(cs)
        e1.record(stream)
        e1.synchronize()
        if s > 0:  # the first pass warms the copy engines
            e2e_ms.append(e0.elapsed_time(e1))
    for s in range(0 if host_entry else e2e_steps + 1):
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
    e2e_step_ms = statistics.median(e2e_ms)
    h2d = sum(2 * (M * K + N * K) + (c_bytes * M * N if fused else 0) for (M, N, K) in shapes)
    d2h = sum(c_bytes * M * N for (M, N, K) in shapes)

    cpu = None
    if not args.no_cpu_baseline:
        rate, cores, sample, secs = oracle_sample_rate(shapes, args.cpu_seconds, ab=ab)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": (f"{sample} ({secs:.1f} s of oracle work; rows not timed "
                          "are estimated from the sample's per-row time plus the "
                          "calibrated fixed cost of decoding B)")}
    roofline = {
        "bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 1),
        "peak": peak_tflops, "unit": "TFLOP/s", "frac": round(achieved / peak_tflops, 4),
        "peak_source": f"{peak_src} x fp16/bf16 nominal ratio 1 (of measured)",
        "traffic": committed_traffic(dom_name, dom["shape"]),
        "traffic_shape": shape_name(dom["shape"]),
        "launches": dom["launches"],
        "frac_vs_sustained": round(achieved / peak_sustained, 4),
        "peak_sustained": peak_sustained,
        "pipe_ceiling": ceiling, "pipe_ceiling_source": ceiling_src,
        "frac_vs_pipe_ceiling": round(achieved / ceiling, 4) if ceiling else None,
    }
    if ktimes is not None and dom["kernel_us"] > 0:
        roofline["achieved_kernel_time"] = round(
            dom["kernel_flops"] / (dom["kernel_us"] * 1e-6) / 1e12, 1)
    line = {
        "metric": METRIC, "value": round(float(value), 2), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ab, "data": "synthetic",
        "config": workload_config(args, shapes),
        "timing": {
            "calls_per_step": {shape_name(s): r for s, r in zip(shapes, reps)},
            "l2": "flushed between calls (256 MiB write), each call timed alone",
            "events": ("CUDA events on the launching stream around each call; a GPU-side "
                       "spin ahead of the start event hides host enqueue latency"),
            "kernel_time": ktime_note,
            "e2e": ("every step: each shape through wgemm_f16f32_host (A and B from pinned "
                    "host memory, C back to pinned host memory; A up in row panels and B "
                    "in blocks of its rows, each GEMM piece starting as its operands "
                    "land, C down piece by piece), each shape on a stream of its own; "
                    "timed from the step's start to the last download" if host_entry else
                    "every step: A and B uploaded from pinned host memory, the call, C "
                    "downloaded; uploads and downloads on two copy streams, pipelined "
                    "across the step's shapes; timed from the first upload to the last "
                    "download"),
        },
        "shapes": per_shape,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_value(float(flops.sum()), e2e_step_ms), 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "wall_s_timed": round(t_wall, 3),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1, help="must be 1: the bench runs one GPU")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="all")
    ap.add_argument("--shape", metavar="MxNxK",
                    help="time this one shape instead of a named workload")
    ap.add_argument("--calls", type=int, default=0,
                    help="calls of every shape per step (default: by shape size)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="oracle time budget of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernel-time", action="store_true",
                    help="skip the CUPTI kernel-time pass")
    ap.add_argument("--config", metavar="NAME",
                    help="force this kernel configuration (profiling; default: the per-shape choice)")
    ap.add_argument("--mode", type=int, default=-1,
                    help="with --config: K decomposition (0 data parallel, 1 split-K, 2 stream-K, "
                         "3 waves + stream-K tail, 4 stream-K with zeroing first)")
    ap.add_argument("--splits", type=int, default=1, help="with --config: split-K ways")
    ap.add_argument("--no-cooperative", action="store_true",
                    help="launch K-split grids without the cooperative attribute (for ncu, which "
                         "runs each kernel alone and cannot profile cooperative launches)")
    ap.add_argument("--types", choices=sorted(TYPES), default="f16f32",
                    help="operand and C types (the measured product is f16f32)")
    ap.add_argument("--values", choices=["uniform", "int"], default="uniform",
                    help="operand values: uniform[-1,1] (the metric) or the integer copy")
    ap.add_argument("--epilogue", choices=["plain", "fused"], default="plain",
                    help="fused: D = A·Bᵀ + D + bias through the alpha/beta/bias epilogue")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    why = single_gpu_only(args)
    if why:
        ap.error(why)
    if args.calls < 0:
        ap.error("--calls wants a count >= 0")
    if args.config and args.epilogue == "fused":
        ap.error("--config forces the plain product")
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
