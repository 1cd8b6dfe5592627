"""GPU kernel times from CUPTI activity records, for the bench.

"SASS-Level Kernel Generation for Blackwell", section "How we measured",
reports each call's GPU kernel time (CUPTI), the median over the last calls.
This module wraps the recorder `libwgemm_ktime.so` (csrc/ktime_cupti.cpp):

    rec = KernelTimes()          # raises KernelTimesUnavailable with the reason
    rec.start()
    ... launches ...
    rec.stop()
    rec.records()                # [(name, start_ns, end_ns, stream), ...] by start time

Measurement tooling only: the GEMM library never uses it.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build


class KernelTimesUnavailable(RuntimeError):
    pass


class KernelTimes:
    def __init__(self):
        if os.environ.get("CUDA_INJECTION64_PATH"):
            # Another profiler (ncu) is attached through the injection hook.
            raise KernelTimesUnavailable("a profiler is attached (CUDA_INJECTION64_PATH)")
        path = _build.build_ktime()
        if path is None:
            raise KernelTimesUnavailable("CUPTI not found in the CUDA toolkit")
        lib = ctypes.CDLL(path)
        ull = ctypes.c_ulonglong
        lib.wkt_start.restype = ctypes.c_int
        lib.wkt_stop.restype = ctypes.c_int
        lib.wkt_flush.restype = ctypes.c_int
        lib.wkt_count.restype = ctypes.c_longlong
        lib.wkt_get.argtypes = [ctypes.c_longlong, ctypes.POINTER(ull), ctypes.POINTER(ull),
                                ctypes.POINTER(ctypes.c_uint), ctypes.c_char_p, ctypes.c_int]
        lib.wkt_get.restype = ctypes.c_int
        lib.wkt_dropped.restype = ull
        lib.wkt_error_string.argtypes = [ctypes.c_int]
        lib.wkt_error_string.restype = ctypes.c_char_p
        self._lib = lib

    def _check(self, rc: int, what: str):
        if rc != 0:
            msg = self._lib.wkt_error_string(rc).decode(errors="replace")
            raise KernelTimesUnavailable(f"{what}: CUPTI error {rc} ({msg})")

    def start(self):
        self._lib.wkt_clear()
        self._check(self._lib.wkt_start(), "enable")

    def stop(self):
        self._check(self._lib.wkt_stop(), "flush")

    def dropped(self) -> int:
        return int(self._lib.wkt_dropped())

    def records(self):
        """Every recorded kernel as (name, start_ns, end_ns, stream), by start."""
        n = self._lib.wkt_count()
        out = []
        s, e = ctypes.c_ulonglong(), ctypes.c_ulonglong()
        st = ctypes.c_uint()
        buf = ctypes.create_string_buffer(512)
        for i in range(n):
            if self._lib.wkt_get(i, ctypes.byref(s), ctypes.byref(e), ctypes.byref(st), buf,
                                 len(buf)) == 0:
                out.append((buf.value.decode(errors="replace"), s.value, e.value, st.value))
        out.sort(key=lambda r: r[1])
        return out
