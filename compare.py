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
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="all")
    ap.add_argument("--rounds", type=int, default=20)
    ap.add_argument("--warm", action="store_true",
                    help="warm L2, synchronised calls, arms in blocks")
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
        for idx, (M, N, K) in enumerate(bench.WORKLOADS[args.workload]):
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
                row.update({"ours_us_kernel": round(ko, 3), "cublas_us_kernel": round(kr, 3),
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
        "workload": args.workload, "rounds": args.rounds, "cublas_output": ref_out,
        "protocol": "warm L2, synchronised calls" if args.warm else "L2 flushed, gated calls",
        "geomean_speedup": round(statistics.geometric_mean(ratios), 3),
        "shapes_faster": sum(1 for x in ratios if x > 1.0), "shapes": len(ratios),
        "torch": torch.__version__, "clocks": clocks.summary()}}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
