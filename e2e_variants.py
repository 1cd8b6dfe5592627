"""The bench's end-to-end step under variants of the host-buffer call: a
measurement, not a product path.

The step is bench.py's end-to-end loop: every shape of the workload through
`wgemm_f16f32_host` (A and B from pinned host memory, C back to pinned host
memory), timed with CUDA events from the step's start to the last download,
after the bench's L2 flush. The variants are the number of caller streams
(2, the shapes alternating, or one per shape as in the bench) and the number
of blocks B's rows go up in (1 or 2 forced through the library's test hook
`wgemm_debug_set_host_blocks`, or the library's rule). The variants run in
alternating rounds, `--steps` timed steps each after one untimed one. Then
one call of the largest shape alone, timed the same way for each block
count.

    python e2e_variants.py [--workload all] [--rounds 4] [--steps 3]

Prints one JSON line per variant (median step ms, min, max, TFLOP/s of the
step) and one per block count of the lone call.
"""
from __future__ import annotations

import argparse
import json
import statistics
import sys

import bench

STREAMS = (2, 0)  # 0: one stream per shape
BLOCKS = (1, 2, 0)  # 0: the library's rule


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", choices=sorted(bench.WORKLOADS), default="all")
    ap.add_argument("--rounds", type=int, default=4)
    ap.add_argument("--steps", type=int, default=3)
    args = ap.parse_args(argv)
    if args.rounds < 1 or args.steps < 1:
        ap.error("--rounds and --steps must be at least 1")
    shapes = bench.WORKLOADS[args.workload]
    if not all(K % 8 == 0 and N % 4 == 0 for (M, N, K) in shapes):
        ap.error("the host call's device layout needs K % 8 == 0 and N % 4 == 0")

    import torch
    from dense_fp16_gemm_02_gb300 import build, inputs, wgemm

    if not torch.cuda.is_available():
        print("e2e_variants: needs a CUDA device", file=sys.stderr)
        return 2
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    build.build()
    lib = wgemm.load()
    data = []
    for i, (M, N, K) in enumerate(shapes):
        A, B = inputs.gemm_operands(M, N, K, seed=1000 + i, kind="uniform")
        hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
        hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
        dA = torch.empty(hA.shape, dtype=hA.dtype, device=dev)
        dB = torch.empty(hB.shape, dtype=hB.dtype, device=dev)
        dC = torch.empty((M, N), dtype=torch.float32, device=dev)
        data.append((hA, hB, hC, dA, dB, dC))
    flush = torch.empty(bench.FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    streams = [torch.cuda.Stream(device=dev) for _ in shapes]
    main_stream = torch.cuda.current_stream()

    def step(n_streams, ids):
        flush.fill_(0.0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main_stream)
        for cs in streams[:n_streams]:
            cs.wait_event(e0)
        for n, i in enumerate(ids):
            M, N, K = shapes[i]
            hA, hB, hC, dA, dB, dC = data[i]
            cs = streams[n % n_streams]
            rc = wgemm.wgemm_f16f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N, K, K,
                                         K, N, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                                         cs.cuda_stream)
            if rc != 0:
                raise RuntimeError(f"wgemm_f16f32_host failed: {wgemm.status_string(rc)}")
        for cs in streams[:n_streams]:
            main_stream.wait_stream(cs)
        e1.record(main_stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    every = list(range(len(shapes)))
    largest = max(every, key=lambda i: 2.0 * shapes[i][0] * shapes[i][1] * shapes[i][2])
    variants = [(s, b) for s in STREAMS for b in BLOCKS]
    times = {v: [] for v in variants}
    lone = {b: [] for b in BLOCKS}
    try:
        for rnd in range(args.rounds):
            for v in (variants if rnd % 2 == 0 else variants[::-1]):
                n_streams = v[0] or len(shapes)
                lib.wgemm_debug_set_host_blocks(v[1])
                step(n_streams, every)
                times[v] += [step(n_streams, every) for _ in range(args.steps)]
            for b in BLOCKS:
                lib.wgemm_debug_set_host_blocks(b)
                step(1, [largest])
                lone[b] += [step(1, [largest]) for _ in range(args.steps)]
    finally:
        lib.wgemm_debug_set_host_blocks(0)
    status = wgemm.wgemm_check(main_stream.cuda_stream)
    if status != 0:
        print(f"e2e_variants: device status {wgemm.status_string(status)}", file=sys.stderr)
        return 1
    flops = sum(2.0 * M * N * K for (M, N, K) in shapes)
    name = lambda b: "rule" if b == 0 else b
    for (s, b), ts in times.items():
        med = statistics.median(ts)
        print(json.dumps({"workload": args.workload,
                          "caller_streams": "one per shape" if s == 0 else s,
                          "b_blocks": name(b), "step_ms": round(med, 3),
                          "min_ms": round(min(ts), 3), "max_ms": round(max(ts), 3),
                          "tflops": round(flops / med / 1e9, 1), "steps": len(ts)}))
    for b, ts in lone.items():
        print(json.dumps({"shape": bench.shape_name(shapes[largest]), "b_blocks": name(b),
                          "call_ms": round(statistics.median(ts), 3), "calls": len(ts)}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
