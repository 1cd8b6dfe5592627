"""The library beside cuBLAS on the same shapes: a comparison, not a product path.

For every shape of a bench workload, the product call (`wgemm_f16f32`,
fp16 A and B, fp32 C) and cuBLAS through `torch.mm(A, Bᵀ, out_dtype=float32)`
(fp16 in, fp32 accumulate and out; the same contraction) are timed call by
call, interleaved as W, ref, ref, W. Every call follows the bench's L2
flush (a 256 MiB write) and GPU-side gate, and is bracketed by CUDA events
on the launching stream. Where this torch has no `out_dtype` for mm, the
cuBLAS arm writes fp16 C (two bytes less per element) and says so.

    python compare.py [--workload all] [--rounds 20]

Prints one JSON line per shape (medians, TFLOP/s of both, and the ratio)
and one summary line. The same checks as the bench guard the comparison:
both arms' results on the shape are compared on a sample of rows.

With `--warm` the calls run the way "SASS-Level Kernel Generation for
Blackwell" (section "How we measured") timed its own: no L2 flush and no
gate, each call followed by a device synchronisation, per shape first
3 + `rounds` calls of the library and then 3 + `rounds` of cuBLAS (the row
check is skipped). Event times then include the launch. With `--cupti` as
well, each call's GPU kernel time comes from the CUPTI recorder (a cuBLAS
call's kernels summed; a marker kernel separates the calls), median over the
timed calls: the pages' own measure. Without it, kernel-only times come from
an ncu launch list of the same command taken with `--cache-control none`,
which `ncu_summary warm <csv> <this output>` turns into a table.

With `--energy` the arms run in blocks of consecutive flushed calls (about
half a second of GEMM time each, no gate: the GPU stays busy, as in a long
run of large GEMMs), the arms' blocks alternating for `rounds` rounds. Each
block reads the GPU's energy counter (NVML, read only) before and after:
joules per call, the mean power and the median time per call (events; the
first third of a block left out while the clock settles). `--configs`
adds arms that force a library configuration. Under the 1.4 kW power cap
a call's energy, not its lone-call time, sets how fast it runs back to back.

`--shape MxNxK` runs one shape instead of a workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="all")
    ap.add_argument("--rounds", type=int, default=20)
    ap.add_argument("--warm", action="store_true",
                    help="warm L2, synchronised calls, arms in blocks")
    ap.add_argument("--shape", metavar="MxNxK", help="one shape instead of a workload")
    ap.add_argument("--energy", action="store_true",
                    help="blocks of back-to-back calls per arm: joules and µs per call")
    ap.add_argument("--configs", default="",
                    help="with --energy: comma-separated library configurations as extra arms")
    ap.add_argument("--cupti", action="store_true",
                    help="with --warm: also each call's kernel time from CUPTI (a cuBLAS call's "
                         "kernels summed), the median over the timed calls")
    args = ap.parse_args(argv)

    import torch
    sys.path.insert(0, ROOT)
    import bench
    from dense_fp16_gemm_02_gb300 import build, inputs, ktime, wgemm
    from dense_fp16_gemm_02_gb300.clocks import ClockSampler
    if args.cupti and not args.warm:
        ap.error("--cupti goes with --warm")
    if args.energy and (args.warm or args.cupti):
        ap.error("--energy runs alone")
    if args.configs and not args.energy:
        ap.error("--configs goes with --energy")
    if args.shape:
        shapes = [tuple(int(v) for v in args.shape.lower().split("x"))]
    else:
        shapes = bench.WORKLOADS[args.workload]
    if args.energy:
        return energy(args, shapes)
    rec = ktime.KernelTimes() if args.cupti else None

    build.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    flush = torch.empty(bench.FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    try:
        probe = torch.zeros((8, 8), dtype=torch.float16, device="cuda")
        torch.mm(probe, probe.t(), out_dtype=torch.float32)
        ref_out = "f32"
    except (TypeError, RuntimeError):
        ref_out = "f16"

    rows = []
    with ClockSampler(0) as clocks:
        clocks.mark_start()
        for idx, (M, N, K) in enumerate(shapes):
            A, B = inputs.gemm_operands(M, N, K, seed=1000 + idx, kind="uniform")
            dA = torch.from_numpy(A).cuda()
            dB = torch.from_numpy(B).cuda()
            del A, B
            C = torch.empty((M, N), dtype=torch.float32, device="cuda")
            Bt = dB.t()

            def ours():
                rc = wgemm.wgemm_f16f32(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K,
                                        K, N, h)
                if rc != 0:
                    raise RuntimeError(wgemm.status_string(rc))

            def ref():
                if ref_out == "f32":
                    return torch.mm(dA, Bt, out_dtype=torch.float32)
                return torch.mm(dA, Bt)

            def timed(fn):
                flush.fill_(0.0)
                torch.cuda._sleep(bench.GATE_CYCLES)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                out = fn()
                e1.record(stream)
                return (e0, e1), out

            def timed_warm(fn):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize()
                return e0, e1

            ev = {"ours": [], "ref": []}
            kt = {"ours": [], "ref": []}
            knames = {"ours": set(), "ref": set()}
            if args.warm:
                for arm, fn in (("ours", ours), ("ref", ref)):
                    if rec is not None:
                        rec.start()
                    for r in range(3 + args.rounds):
                        e = timed_warm(fn)
                        if r >= 3:
                            ev[arm].append(e)
                        if rec is not None:  # a marker kernel after every call
                            torch.cuda._sleep(16)
                            torch.cuda.synchronize()
                    if rec is not None:
                        rec.stop()
                        # Each call's kernels lie between two markers (the
                        # sleep kernel); a cuBLAS call may launch several.
                        calls, cur = [], 0.0
                        for name, t0, t1, _ in rec.records():
                            if "sleep" in name or "spin" in name:
                                calls.append(cur)
                                cur = 0.0
                            else:
                                cur += (t1 - t0) * 1e-3
                                knames[arm].add(name[:120])
                        kt[arm] = calls[3:]
            else:
                for _ in range(3):  # warm-up, both arms
                    timed(ours)
                    timed(ref)
                for _ in range(args.rounds):  # W, ref, ref, W
                    for arm, fn in (("ours", ours), ("ref", ref), ("ref", ref), ("ours", ours)):
                        e, _ = timed(fn)
                        ev[arm].append(e)
            torch.cuda.synchronize()
            if wgemm.wgemm_check(h) != 0:
                raise RuntimeError(f"device status: {wgemm.wgemm_last_device_error()}")
            err = None
            if not args.warm:
                # The two arms compute the same contraction: compare a sample of rows.
                rsel = torch.linspace(0, M - 1, steps=min(M, 64)).long().cuda()
                Cr = ref().float()
                scale = (dA[rsel].float().abs() @ dB.float().abs().t())
                err = float(((C[rsel] - Cr[rsel]).abs() / (scale + 1e-6)).max())
                del Cr
            us = {a: statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev[a])
                  for a in ev}
            fl = 2.0 * M * N * K
            row = {"shape": f"{M}x{N}x{K}", "ours_us": round(us["ours"], 3),
                   "cublas_us": round(us["ref"], 3),
                   "ours_tflops": round(fl / us["ours"] / 1e6, 1),
                   "cublas_tflops": round(fl / us["ref"] / 1e6, 1),
                   "speedup": round(us["ref"] / us["ours"], 3),
                   "max_rel_diff_vs_abs_product": err}
            if rec is not None:
                if len(kt["ours"]) != args.rounds or len(kt["ref"]) != args.rounds:
                    raise RuntimeError(f"CUPTI: {len(kt['ours'])} and {len(kt['ref'])} calls "
                                       f"for {args.rounds} rounds")
                ko, kr = statistics.median(kt["ours"]), statistics.median(kt["ref"])
                row.update({"cublas_kernels": sorted(knames["ref"]),
                            "ours_us_kernel": round(ko, 3), "cublas_us_kernel": round(kr, 3),
                            "ours_tflops_kernel": round(fl / ko / 1e6, 1),
                            "cublas_tflops_kernel": round(fl / kr / 1e6, 1),
                            "speedup_kernel": round(kr / ko, 3)})
            rows.append(row)
            print(json.dumps(row), flush=True)
            del dA, dB, Bt, C
            torch.cuda.empty_cache()
        clocks.mark_stop()
    ratios = [r["speedup"] for r in rows]
    kratios = [r["speedup_kernel"] for r in rows if "speedup_kernel" in r]
    print(json.dumps({"summary": {
        "geomean_speedup_kernel": (round(statistics.geometric_mean(kratios), 3) if kratios
                                   else None),
        "workload": args.shape or args.workload, "rounds": args.rounds, "cublas_output": ref_out,
        "protocol": "warm L2, synchronised calls" if args.warm else "L2 flushed, gated calls",
        "geomean_speedup": round(statistics.geometric_mean(ratios), 3),
        "shapes_faster": sum(1 for x in ratios if x > 1.0), "shapes": len(ratios),
        "torch": torch.__version__, "clocks": clocks.summary()}}), flush=True)
    return 0


def energy(args, shapes) -> int:
    import torch
    import bench
    from dense_fp16_gemm_02_gb300 import build, inputs, wgemm
    from dense_fp16_gemm_02_gb300.clocks import ClockSampler, EnergyCounter

    build.build()
    torch.cuda.set_device(0)
    meter = EnergyCounter()
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    flush = torch.empty(bench.FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    forced = [c for c in args.configs.split(",") if c]
    for c in forced:
        wgemm.config_id(c)  # unknown names fail here, before any timing
    summary = []
    torch.cuda.synchronize()
    time.sleep(0.5)
    j0, t0 = meter.joules(), time.perf_counter()
    time.sleep(2.0)
    idle_w = (meter.joules() - j0) / (time.perf_counter() - t0)
    with ClockSampler(0) as clocks:
        clocks.mark_start()
        for idx, (M, N, K) in enumerate(shapes):
            A, B = inputs.gemm_operands(M, N, K, seed=1000 + idx, kind="uniform")
            dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
            del A, B
            C = torch.empty((M, N), dtype=torch.float32, device="cuda")
            Bt = dB.t()

            def arm_fn(arm):
                if arm == "cublas":
                    return lambda: torch.mm(dA, Bt, out_dtype=torch.float32)
                cid = None if arm == "library" else wgemm.config_id(arm)

                def f():
                    if cid is None:
                        rc = wgemm.wgemm_f16f32(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N,
                                                K, K, K, N, h)
                    else:
                        rc = wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(),
                                                       C.data_ptr(), M, N, K, K, K, N, cid, 0, 1,
                                                       h)
                    if rc != 0:
                        raise RuntimeError(wgemm.status_string(rc))
                return f

            arms = ["library", "cublas"] + forced
            fns = {a: arm_fn(a) for a in arms}
            # Calls per block from one timed call of the library.
            for _ in range(3):
                flush.fill_(0.0)
                fns["library"]()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fns["library"]()
            e1.record(stream)
            torch.cuda.synchronize()
            calls = max(30, int(0.5e6 / max(e0.elapsed_time(e1) * 1e3, 1.0)))
            res = {a: {"j": [], "us": [], "w": []} for a in arms}
            for r in range(args.rounds):
                order = arms if r % 2 == 0 else arms[::-1]
                for a in order:
                    evs = [(torch.cuda.Event(enable_timing=True),
                            torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
                    torch.cuda.synchronize()
                    j0 = meter.joules()
                    t0 = time.perf_counter()
                    for i in range(calls):
                        flush.fill_(float(i))
                        evs[i][0].record(stream)
                        fns[a]()
                        evs[i][1].record(stream)
                    torch.cuda.synchronize()
                    t1 = time.perf_counter()
                    # The counter lags the work by up to one update: read it
                    # after a pause and take out the pause's idle energy.
                    time.sleep(0.2)
                    work_j = meter.joules() - j0 - idle_w * (time.perf_counter() - t1)
                    ts = [x.elapsed_time(y) * 1e3 for x, y in evs]
                    res[a]["us"].append(statistics.median(ts[calls // 3:]))
                    res[a]["j"].append(work_j / calls)
                    res[a]["w"].append(work_j / (t1 - t0))
                    time.sleep(0.3)
            if wgemm.wgemm_check(h) != 0:
                raise RuntimeError(f"device status: {wgemm.wgemm_last_device_error()}")
            for a in arms:
                row = {"shape": f"{M}x{N}x{K}", "arm": a,
                       "config": (wgemm.config_name(wgemm.wgemm_select(M, N, K)[0])
                                  if a == "library" else a),
                       "calls_per_block": calls, "blocks": args.rounds,
                       "us_per_call": round(statistics.median(res[a]["us"]), 1),
                       "joules_per_call": round(statistics.median(res[a]["j"]), 4),
                       "watts": round(statistics.median(res[a]["w"]), 1),
                       "tflops": round(2.0 * M * N * K / statistics.median(res[a]["us"]) / 1e6, 1)}
                summary.append(row)
                print(json.dumps(row), flush=True)
            del dA, dB, Bt, C
            torch.cuda.empty_cache()
        clocks.mark_stop()
    print(json.dumps({"summary": {"protocol": "blocks of back-to-back flushed calls, energy "
                                              "from the NVML counter (flush included)",
                                  "energy_device": meter.device, "idle_watts": round(idle_w, 1),
                                  "rounds": args.rounds,
                                  "torch": torch.__version__, "clocks": clocks.summary()}}),
          flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
