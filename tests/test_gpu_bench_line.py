"""bench.py's main arm on the GPU: one JSON line that keeps the measurement contract.

A short run (few steps, no cuBLAS, no workload pass) through the same code as the default
one: the headline value is the 4096^3 GEMM's whole-job TFLOP/s, the roofline object divides
it by the measured peak, the end-to-end figure moves A and B in and D out every step, every
timed step is one launch of this library's kernel, and the cpu_baseline leg times the oracle
after checking sampled outputs against it.  Without that leg the oracle is not run at all.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_main_arm_prints_the_contract_line():
    steps, warmup = 50, 3
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", str(steps), "--warmup",
                          str(warmup), "--no-cublas", "--no-workloads", "--e2e-steps", "5",
                          "--sustained-seconds", "0.5"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert (d["metric"], d["unit"], d["higher_is_better"], d["scaling"]) == (bench.METRIC, bench.UNIT, True, "weak")
    assert (d["n_gpus"], d["steps"], d["warmup"], d["dtype"], d["data"]) == (1, steps, warmup, "f16", "synthetic")
    assert d["config"]["workload"] == bench.WORKLOAD and d["vs_baseline"] is None
    M = N = K = 4096
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["value"] == pytest.approx(2.0 * M * N * K / (d["ms_per_step"] * 1e-3) / 1e12, rel=1e-6)
    r = d["roofline"]
    assert (r["bound"], r["unit"]) == ("tensor", "TFLOP/s") and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9)
    # 50 launches of ~80 us are a burst: set against the measured burst peak
    timed_s = steps * d["ms_per_step"] / 1e3
    assert r["peak_regime"] == ("sustained" if timed_s >= bench.SUSTAINED_REGION_S else "burst")
    assert r["frac_of_burst"] == pytest.approx(r["achieved"] / bench.measured_peak()[0], rel=1e-9)
    assert r["traffic"] is None or r["traffic"] > 0
    e = d["e2e"]
    assert e["unit"] == d["unit"] and 0 < e["value"] < d["value"]
    assert (e["h2d_bytes_per_step"], e["d2h_bytes_per_step"]) == (2 * (M * K + N * K), 2 * M * N)
    assert d["gpu_launches"] == steps
    assert d["parity_vs_oracle"]["pass"] is True  # the guard's sampled outputs against the oracle
    assert r["stated_peak"] == 2500.0 and r["frac_of_stated_peak"] == pytest.approx(r["achieved"] / 2500.0)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["unit"] == d["unit"] and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["cpu_model"]
    c = d["clocks"]
    assert set(c) >= {"sm_mhz", "sm_max_mhz", "reasons", "note"}
    # a timed region shorter than the sampling interval still gets the nearest sample
    assert c["sm_mhz"] is not None and c["sm_max_mhz"] is not None, c
    s = d["sustained"]
    assert s["value"] > 0 and s["unit"] == d["unit"] and len(s["windows"]) == 2
    assert all(w["gemms"] > 0 and w["sm_mhz"] for w in s["windows"])


def test_without_the_cpu_baseline_leg_the_oracle_is_not_run():
    env = dict(os.environ, PYTHONPATH=ROOT)
    code = ("import sys, runpy; sys.argv = ['bench.py', '--steps', '5', '--warmup', '3', '--no-cublas', "
            "'--no-cpu-baseline', '--e2e-steps', '2']; runpy.run_path('bench.py', run_name='__main__'); "
            "print('ORACLE_LOADED' if any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules) "
            "else 'ORACLE_ABSENT')")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    assert out.stdout.strip().splitlines()[-1] == "ORACLE_ABSENT"
    d = json.loads([ln for ln in out.stdout.splitlines() if ln.startswith("{")][0])
    assert d["parity_vs_oracle"] is None and "cpu_baseline" not in d
    assert all(w["parity_vs_oracle"] is None and "oracle" not in w for w in d["workloads"])
