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


class EnergyCounterUnavailable(RuntimeError):
    pass


class EnergyCounter:
    """The GPU's total-energy counter (NVML, millijoules since the driver
    loaded), read only. The device is the one torch calls cuda:0, found by
    its PCI address; where torch does not give that address, NVML must see
    exactly one GPU."""

    def __init__(self):
        import ctypes

        import torch
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError as e:
            raise EnergyCounterUnavailable(f"NVML not found: {e}") from e
        if nv.nvmlInit_v2() != 0:
            raise EnergyCounterUnavailable("nvmlInit failed")
        handle = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(0)
        bus = getattr(props, "pci_bus_id", None)
        if bus is not None:
            pci = (f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:"
                   f"{getattr(props, 'pci_device_id', 0):02x}.0")
            rc = nv.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(handle))
            self.device = f"PCI {pci}"
        else:
            count = ctypes.c_uint()
            nv.nvmlDeviceGetCount_v2(ctypes.byref(count))
            if count.value != 1:
                raise EnergyCounterUnavailable(f"NVML sees {count.value} GPUs and torch gives "
                                               "no PCI address")
            rc = nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(handle))
            self.device = "NVML index 0 (the only GPU)"
        if rc != 0:
            raise EnergyCounterUnavailable(f"no NVML handle for {self.device} (error {rc})")
        self._nv, self._handle, self._ct = nv, handle, ctypes

    def joules(self) -> float:
        mj = self._ct.c_ulonglong()
        rc = self._nv.nvmlDeviceGetTotalEnergyConsumption(self._handle, self._ct.byref(mj))
        if rc != 0:
            raise EnergyCounterUnavailable(f"nvmlDeviceGetTotalEnergyConsumption: error {rc}")
        return mj.value / 1000.0
