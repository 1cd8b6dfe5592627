"""Tensor-pipe ceiling of the GPU for the MMA shapes the kernels use.

Builds `peak/tensor_peak.cu` (sm_103a) and runs it under clock sampling:
every CTA or CTA pair issues back-to-back tcgen05.mma on operands resident in
shared memory, with no global traffic in the timed loop. Prints one JSON line
per MMA shape, then one with the SM clock seen during the run.

    python -m dense_fp16_gemm_02_gb300.peak [iterations]

With `--interference` it builds and runs `peak/mma_interference.cu`
instead: the pair M256 N224 MMA loop while four more warps of every CTA
make one kind of traffic (global stores, the register-store epilogue's
pattern, shared-memory stores or loads, TMEM loads, bulk copies into shared
memory), one JSON line per kind with the MMA rate and the traffic's rate.

    python -m dense_fp16_gemm_02_gb300.peak --interference [iterations]
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

from . import build as _build
from .clocks import ClockSampler

HERE = os.path.dirname(os.path.abspath(__file__))
PROGRAMS = ("tensor_peak", "mma_interference")


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


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    name = "tensor_peak"
    if argv and argv[0] == "--interference":
        name, argv = "mma_interference", argv[1:]
    exe = build_peak(name)
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
