"""Clock and power record of a timed region: the SM clock, power and throttle reasons, sampled
while the GEMMs run.

Under a long run of dense GEMMs the GPU sits at its power cap and the SM clock follows the
power drawn, so a throughput figure means little without the clock it ran at.  The samples
come from read-only NVML queries in this process (the driver's own library through ctypes;
nothing is set), every millisecond by default so that even a timed region of a few
milliseconds holds samples, or from ``nvidia-smi -lms`` where NVML cannot be loaded.
"""
from __future__ import annotations

import statistics
import subprocess
import threading
import time


class _Nvml:
    """Read-only NVML queries through the driver's own library (ctypes; nothing is set)."""

    SM = 1  # NVML_CLOCK_SM
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int):
        import ctypes

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.SM)

    def _uint(self, fn, *args):
        v = self.ct.c_uint(0)
        return float(v.value) if fn(self.dev, *args, self.ct.byref(v)) == 0 else None

    def sample(self):
        sm = self._uint(self.lib.nvmlDeviceGetClockInfo, self.SM)
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        bits = self.ct.c_ulonglong(0)
        ok = self.reasons_fn(self.dev, self.ct.byref(bits)) == 0
        reasons = [name for bit, name in self.REASON_BITS.items() if ok and bits.value & bit]
        return sm, self.max_mhz, (mw / 1000.0 if mw is not None else None), reasons

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock, power and throttle reasons sampled (time-stamped) while the benchmark runs:
    in-process NVML queries every `interval_ms` (1 ms by default, so that even a timed region
    of a few milliseconds holds samples), or `nvidia-smi -lms` where NVML cannot be loaded."""

    def __init__(self, gpu_index: int, interval_ms: float = 1.0):
        self.samples: list[tuple[float, tuple]] = []  # (time, (sm_mhz, max_mhz, power_w, reasons))
        self.proc = None
        self.nvml = None
        self.stopping = False
        try:
            self.nvml = _Nvml(gpu_index)
            self.source = "nvml"
            self.interval_s = interval_ms / 1000.0
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            self.nvml = None
        self.source = "nvidia-smi"
        self.interval_s = max(interval_ms, 100) / 1000.0
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", str(int(self.interval_s * 1000))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def _poll(self):
        while not self.stopping:
            self.samples.append((time.time(), self.nvml.sample()))
            time.sleep(self.interval_s)

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        for line in self.proc.stdout:
            p = [x.strip() for x in line.strip().split(",")]
            if len(p) == len(self.FIELDS):
                reasons = [names[i] for i in range(4) if p[4 + i].lower().startswith("active")]
                self.samples.append((time.time(), (num(p[0]), num(p[1]), num(p[2]), reasons)))

    def wait_for_sample(self, after: float, timeout_s: float = 3.0) -> bool:
        """Block until a sample stamped after `after` has arrived (or the timeout): nvidia-smi
        takes a moment to start, and a short timed region may end before the next sample."""
        if self.proc is None and self.nvml is None:
            return False
        t_end = time.time() + timeout_s
        while time.time() < t_end:
            if any(t > after for t, _ in self.samples):
                return True
            time.sleep(0.001)
        return False

    def stop(self):
        self.stopping = True
        if self.nvml is not None:
            self.thread.join(timeout=2)
            self.nvml.close()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        """Clock record of the region [t0, t1] (wall-clock seconds).  A region shorter than the
        sampling interval may hold no sample: then the sample nearest to the region (waiting
        for the next one if none has arrived yet) stands for it, and the note says how far
        from the region it was taken."""
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:
            self.wait_for_sample(t1, timeout_s=3 * self.interval_s + 1.0)
            if self.samples:
                mid = 0.5 * (t0 + t1)
                t, p = min(self.samples, key=lambda tp: abs(tp[0] - mid))
                gap_ms = (t0 - t if t < t0 else t - t1) * 1e3
                side = "before the region's start" if t < t0 else "after the region's end"
                inside = [p]
                note = (f"timed region ({(t1 - t0) * 1e3:.1f} ms) shorter than the {self.interval_s * 1e3:.0f} ms "
                        f"sampling interval: the nearest sample, {gap_ms:.0f} ms {side}")
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no clock sample arrived",
                    "source": self.source}
        sm = [p[0] for p in inside if p[0] is not None]
        power = [p[2] for p in inside if p[2] is not None]
        reasons = sorted({r for p in inside for r in p[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": inside[0][1],
                "reasons": reasons, "power_w_max": max(power) if power else None, "samples": len(inside),
                "note": note, "source": self.source}
