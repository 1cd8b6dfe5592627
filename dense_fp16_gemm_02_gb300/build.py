"""Builds libwgemm.so in-tree (dense_fp16_gemm_02_gb300/_build/) with nvcc.

Each translation unit is compiled in parallel for sm_103a only, then linked
into one shared library with the CUDA runtime linked statically. No CMake, no
torch extension builder: plain nvcc.

Beside it, when the toolkit's CUPTI is present, the bench's kernel-time
recorder libwgemm_ktime.so (csrc/ktime_cupti.cpp, g++ against libcupti). The
GEMM library does not depend on it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libwgemm.so")
SOURCES = ["wgemm_host.cu", "inst_single.cu", "inst_pair.cu", "inst_pair2.cu",
           "inst_multicast.cu", "inst_clc.cu", "inst_out16_a.cu", "inst_out16_b.cu",
           "inst_fused.cu", "inst_rowmc.cu"]
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-DNDEBUG", "-Xcompiler", "-fPIC",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
# WGEMM_CHECKED=1 in the environment builds the index-checking debug variant
# into a separate directory (dense_fp16_gemm_02_gb300/_build_checked).
if os.environ.get("WGEMM_CHECKED") == "1":
    FLAGS.append("-DWGEMM_CHECKED=1")
    BUILD = os.path.join(HERE, "_build_checked")
    LIB = os.path.join(BUILD, "libwgemm.so")
# WGEMM_TRACE=1 builds the timeline-tracing variant (dense_fp16_gemm_02_gb300/_build_trace).
if os.environ.get("WGEMM_TRACE") == "1":
    FLAGS.append("-DWGEMM_TRACE=1")
    BUILD = os.path.join(HERE, "_build_trace")
    LIB = os.path.join(BUILD, "libwgemm.so")


def _headers() -> list[str]:
    out = []
    for d, _, files in os.walk(CSRC):
        out += [os.path.join(d, f) for f in files if f.endswith((".h", ".cuh", ".inc"))]
    out.append(os.path.join(ROOT, "include", "wgemm.h"))
    return out


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src)] + _headers()
    if _stale(obj, deps) or verbose_ptxas:
        cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj + ".tmp"]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
        os.replace(obj + ".tmp", obj)
    return obj


KTIME_SRC = os.path.join(CSRC, "ktime_cupti.cpp")
KTIME_LIB = os.path.join(BUILD, "libwgemm_ktime.so")


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home:
        return home
    nvcc = shutil.which(NVCC)
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def cupti_paths():
    """(include dir, library dir) of the toolkit's CUPTI, or None."""
    home = _cuda_home()
    incs = [os.path.join(home, "extras", "CUPTI", "include"), os.path.join(home, "include")]
    libs = [os.path.join(home, "extras", "CUPTI", "lib64"), os.path.join(home, "lib64")]
    tdir = os.path.join(home, "targets")
    if os.path.isdir(tdir):
        for t in sorted(os.listdir(tdir)):
            incs.append(os.path.join(tdir, t, "include"))
            libs.append(os.path.join(tdir, t, "lib"))
    inc = next((d for d in incs if os.path.exists(os.path.join(d, "cupti.h"))), None)
    lib = next((d for d in libs if os.path.exists(os.path.join(d, "libcupti.so"))), None)
    return (inc, lib) if inc and lib else None


def build_ktime() -> str | None:
    """Compile the CUPTI kernel-time recorder; None when CUPTI is absent."""
    paths = cupti_paths()
    if paths is None:
        return None
    inc, lib = paths
    os.makedirs(BUILD, exist_ok=True)
    if not _stale(KTIME_LIB, [KTIME_SRC]):
        return KTIME_LIB
    tmp = KTIME_LIB + f".{os.getpid()}.tmp"
    cmd = [os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-fPIC", "-shared", "-I", inc,
           KTIME_SRC, "-o", tmp, "-L", lib, "-lcupti", f"-Wl,-rpath,{lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"kernel-time recorder build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, KTIME_LIB)
    return KTIME_LIB


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile every translation unit (in parallel) and link libwgemm.so;
    also the kernel-time recorder where CUPTI is present."""
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    if _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    build_ktime()
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
