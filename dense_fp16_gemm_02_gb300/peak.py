"""Tensor-pipe ceiling of the GPU for the MMA shapes the kernels use.

Builds `peak/tensor_peak.cu` (sm_103a) and runs it under clock sampling:
every CTA or CTA pair issues back-to-back tcgen05.mma on operands resident in
shared memory, with no global traffic in the timed loop. Prints one JSON line
per MMA shape, then one with the SM clock seen during the run.

    python -m dense_fp16_gemm_02_gb300.peak [iterations]
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

from . import build as _build
from .clocks import ClockSampler

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "peak", "tensor_peak.cu")
EXE = os.path.join(_build.BUILD, "tensor_peak")


def build_peak() -> str:
    os.makedirs(_build.BUILD, exist_ok=True)
    deps = [SRC, os.path.join(HERE, "csrc", "sm103", "ptx.cuh"),
            os.path.join(HERE, "csrc", "sm103", "umma_desc.h")]
    if os.path.exists(EXE) and os.path.getmtime(EXE) >= max(os.path.getmtime(d) for d in deps):
        return EXE
    cmd = [_build.NVCC, *_build.ARCH, "-O3", "-std=c++17", "-o", EXE, SRC]
    subprocess.run(cmd, check=True)
    return EXE


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    exe = build_peak()
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
