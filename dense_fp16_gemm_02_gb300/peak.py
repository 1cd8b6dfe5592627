"""Tensor-pipe ceiling of the GPU for the MMA shapes the kernels use.

Builds `peak/tensor_peak.cu` (sm_103a) and runs it under clock sampling:
every CTA or CTA pair issues back-to-back tcgen05.mma on operands resident in
shared memory, with no global traffic in the timed loop. Prints one JSON line
per MMA shape, then one with the SM clock seen during the run.

    python -m dense_fp16_gemm_02_gb300.peak [iterations]

With `--copies` it measures the host-device copy engines instead, the bound
of the bench's end-to-end figure: pinned host memory to the device, back,
and both directions at once on two streams, for 32, 128 and 256 MiB (CUDA
events, median of ten after two warm-ups), one JSON line per size.

    python -m dense_fp16_gemm_02_gb300.peak --copies
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

from . import build as _build
from .clocks import ClockSampler

HERE = os.path.dirname(os.path.abspath(__file__))
PROGRAMS = ("tensor_peak",)


def build_peak(name: str = "tensor_peak") -> str:
    """Compile peak/<name>.cu for sm_103a (when stale); returns the executable."""
    assert name in PROGRAMS
    src = os.path.join(HERE, "peak", name + ".cu")
    exe = os.path.join(_build.BUILD, name)
    os.makedirs(_build.BUILD, exist_ok=True)
    deps = [src, os.path.join(HERE, "csrc", "sm103", "ptx.cuh"),
            os.path.join(HERE, "csrc", "sm103", "umma_desc.h")]
    if os.path.exists(exe) and os.path.getmtime(exe) >= max(os.path.getmtime(d) for d in deps):
        return exe
    cmd = [_build.NVCC, *_build.ARCH, "-O3", "-std=c++17", "-o", exe, src]
    subprocess.run(cmd, check=True)
    return exe


def copy_rates(sizes_mib=(32, 128, 256), reps=10):
    """Host-device copy bandwidths (GB/s) with pinned host buffers."""
    import torch
    dev = torch.device("cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    out = []

    def on_two(first, second):
        """Run two copies at once, one per stream, after the current stream's work."""
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        s1.wait_event(start)
        s2.wait_event(start)
        with torch.cuda.stream(s1):
            first()
        with torch.cuda.stream(s2):
            second()
        for s in (s1, s2):
            e = torch.cuda.Event()
            e.record(s)
            cur.wait_event(e)

    for mib in sizes_mib:
        n = mib << 20
        h_in = torch.empty(n, dtype=torch.uint8).pin_memory()
        h_out = torch.empty(n, dtype=torch.uint8).pin_memory()
        d_in = torch.empty(n, dtype=torch.uint8, device=dev)
        d_out = torch.empty(n, dtype=torch.uint8, device=dev)
        d_in2 = torch.empty(n, dtype=torch.uint8, device=dev)
        h_out2 = torch.empty(n, dtype=torch.uint8).pin_memory()

        def timed(fn):
            ts = []
            for _ in range(reps + 2):
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            ts = sorted(ts[2:])
            return ts[len(ts) // 2] * 1e-3  # s

        def both():
            on_two(lambda: d_in.copy_(h_in, non_blocking=True),
                   lambda: h_out.copy_(d_out, non_blocking=True))

        def two_up():  # two uploads at once: more copy engines, the same link
            on_two(lambda: d_in.copy_(h_in, non_blocking=True),
                   lambda: d_in2.copy_(h_out, non_blocking=True))

        def two_down():
            on_two(lambda: h_out.copy_(d_out, non_blocking=True),
                   lambda: h_out2.copy_(d_in, non_blocking=True))

        out.append({
            "mib": mib,
            "h2d_gbs": round(n / timed(lambda: d_in.copy_(h_in, non_blocking=True)) / 1e9, 1),
            "d2h_gbs": round(n / timed(lambda: h_out.copy_(d_out, non_blocking=True)) / 1e9, 1),
            "both_directions_gbs": round(2 * n / timed(both) / 1e9, 1),
            "h2d_two_streams_gbs": round(2 * n / timed(two_up) / 1e9, 1),
            "d2h_two_streams_gbs": round(2 * n / timed(two_down) / 1e9, 1),
        })
    return out


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    if argv and argv[0] == "--copies":
        for row in copy_rates():
            print(json.dumps(row))
        return 0
    exe = build_peak("tensor_peak")
    with ClockSampler(0) as clocks:
        clocks.mark_start()
        out = subprocess.run([exe, *argv], check=True, capture_output=True, text=True).stdout
        clocks.mark_stop()
    for line in out.splitlines():
        if line.startswith("{"):
            print(line)
    print(json.dumps({"clocks": clocks.summary()}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
