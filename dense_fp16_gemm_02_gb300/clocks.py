"""nvidia-smi clock and throttle sampling of a timed region.

Used by bench.py and the tensor-pipe microbenchmark runner (peak.py): the
SM clock and the throttle reasons seen while the measured work ran.
"""
from __future__ import annotations

import datetime
import statistics
import subprocess
import threading
import time


class ClockSampler:
    """nvidia-smi clock / throttle sampling of the timed region.

    nvidia-smi stamps every sample with its own clock time; the sampler is
    started (and its first sample awaited) before the timed region, the region
    is marked with mark_start() / mark_stop(), and only samples stamped inside
    it are summarised."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None
        self._reader = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.proc = None
            return self
        first = threading.Event()

        def read():
            for line in self.proc.stdout:
                if line.strip():
                    self.lines.append(line.strip())
                    first.set()
        self._reader = threading.Thread(target=read, daemon=True)
        self._reader.start()
        first.wait(timeout=10)  # sampling has begun before the timed region starts
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)  # one more sample period, so the region's last sample lands
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self._reader is not None:
                self._reader.join(timeout=5)

    @staticmethod
    def _stamp(text: str):
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        sm, smax, reasons, outside = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            t = self._stamp(parts[0])
            if (t is not None and self.t_start is not None and self.t_stop is not None
                    and not (self.t_start - 0.05 <= t <= self.t_stop + 0.05)):
                outside += 1
                continue
            try:
                sm.append(float(parts[2]))
                smax = float(parts[3])
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_outside_region": outside}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_outside_region": outside}
