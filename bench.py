#!/usr/bin/env python
"""Benchmark of the sm_103a fp16 GEMM D = A·Bᵀ on the 4096³ headline workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one GEMM over one input set (the whole hot path: one kernel launch).
Prints ONE JSON line (rank 0).  For N > 1 run under torchrun: every rank runs
its own replica on its own GPU (the GEMM has no exchange step), so the scaling
is weak and the value is the total over ranks.

Timing: W untimed warm-up steps, then K steps between a barrier +
synchronize on both sides, measured with CUDA events on the stream the kernel
is launched on.  Inputs and outputs rotate over 4 device copies (384 MiB, above
the 129 MB L2), so every step reads A and B from HBM.  nvidia-smi clocks and
throttle reasons are sampled while the timed region runs.

``--impl reference`` times the CPU oracle (plain C, fp64 accumulation) as it
stands on this machine's host cores, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402
from blackwell_tensor_core_02_gb300.clocks import ClockSampler  # noqa: E402

METRIC = "GEMM TFLOP/s at M=N=K=4096 fp16→fp32 acc; % of GB300 dense fp16 tensor peak"
UNIT = "TFLOP/s"
WORKLOAD = si.HEADLINE
ROTATE = 4
# NVIDIA's published GB300 dense fp16/bf16 tensor figure (5 PFLOP/s with 2:4 sparsity, halved):
# the stated peak the target of >= 70 % refers to
STATED_PEAK_TFLOPS = 2500.0
FALLBACK_PEAK_TFLOPS = 1900.0         # one earlier cuBLAS bf16 measurement on a GB300
# A timed region of back-to-back GEMMs at least this long runs under the power cap, the
# regime of MEASURED_PEAKS.json's sustained figure (a seconds-long cuBLAS loop); a shorter
# one is a burst and is set against the burst figure.
SUSTAINED_REGION_S = 0.25
KERNEL_NAME = "gemm_f16_nt_kernel<2, 1, 256, 128, 1>"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "ncu_gemm_f16_nt_kernel_square_4096.json")


def source_code_only(text: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace collapsed (the sources hold no
    comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(csrc: str | None = None) -> str:
    """Hash of the CUDA sources' code (comments and layout ignored): the ncu traffic figure is
    only valid for the kernel it was taken on."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "blackwell_tensor_core_02_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + source_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None, \
            "measured: MEASURED_PEAKS.json bf16_tflops (cuBLAS bf16 burst); fp16 runs at the bf16 rate"
    except (OSError, KeyError, ValueError):
        return FALLBACK_PEAK_TFLOPS, None, "fallback: 1.9 PFLOP/s bf16 burst from an earlier GB300 measurement"


def ncu_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, or None if absent or stale."""
    try:
        with open(PROFILE_SUMMARY) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, "no ncu summary committed"
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    return int(d["dram_bytes_per_launch"]), d.get("command", "")


# --------------------------------------------------------- rank arithmetic --

def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank sets the job's time)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def roofline_peak(timed_s: float, peak: float, peak_sustained, source: str):
    """The roofline's denominator for a timed region of `timed_s` seconds: the measured
    sustained peak once the region is long enough to run under the power cap, else the
    burst peak.  Returns (peak, regime, source)."""
    if peak_sustained and timed_s >= SUSTAINED_REGION_S:
        return peak_sustained, "sustained", (
            f"measured: MEASURED_PEAKS.json bf16_tflops_sustained (cuBLAS bf16, seconds-long loop under the "
            f"power cap), as this timed region ({timed_s:.2f} s of back-to-back launches) runs under the "
            f"same cap; fp16 runs at the bf16 rate")
    return peak, "burst", source


def whole_job_tflops(flop_per_step: float, steps: int, world: int, elapsed_ms: float) -> float:
    """Total TFLOP/s of `world` replicas that each ran `steps` steps in `elapsed_ms` (max over ranks)."""
    return world * flop_per_step * steps / (elapsed_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ clocks --

DISQUALIFYING_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def needs_remeasure(clocks) -> bool:
    """Whether a timed region's clock record disqualifies the run: a hardware or thermal
    slowdown, or SM clocks far below their maximum with no reason given (a clock lock left
    by someone else).  The power cap (sw_power_cap) is normal for a dense GEMM and is kept."""
    if not clocks or clocks.get("sm_mhz") is None:
        return False
    reasons = set(clocks.get("reasons") or [])
    if reasons & set(DISQUALIFYING_REASONS):
        return True
    top = clocks.get("sm_max_mhz")
    return not reasons and bool(top) and clocks["sm_mhz"] < 0.7 * top


# ------------------------------------------------------------- CPU oracle --

def parity_stats(got, ref) -> dict:
    """How the sampled GPU outputs compare with the oracle's (both fp16 values as float64):
    the tolerance is |got - ref| <= 2^-9 |ref| + 1e-3 per element."""
    err = np.abs(got - ref)
    tol = 2.0 ** -9 * np.abs(ref) + 1e-3
    return {"points": int(got.size), "equal_to_oracle": float(np.mean(got == ref)),
            "max_abs_err": float(err.max()), "worst_fraction_of_tolerance": float((err / tol).max()),
            "pass": bool(np.all(err <= tol))}


def oracle_rows_tflops(A, B, rows: int, threads: int):
    """The oracle as it stands on `rows` full rows of D; returns (TFLOP/s, seconds)."""
    import oracle

    t0 = time.perf_counter()
    oracle.gemm_f16_nt(A[:rows], B, threads=threads)
    dt = time.perf_counter() - t0
    return 2.0 * rows * B.shape[0] * A.shape[1] / dt / 1e12, dt


def oracle_rows_calibrated(A, B, threads: int, target_s: float):
    """Time the oracle on as many full rows of D as take about target_s.  Two-point
    calibration first: each call decodes all of B once (a fixed cost), then costs the same
    per row.  Returns (rows, TFLOP/s, seconds, per-row seconds, fixed seconds)."""
    r1, r2 = min(A.shape[0], threads), min(A.shape[0], 4 * threads)
    _, t1 = oracle_rows_tflops(A, B, r1, threads)
    _, t2 = oracle_rows_tflops(A, B, r2, threads)
    per_row = max((t2 - t1) / max(r2 - r1, 1), 1e-9)
    fixed = max(t1 - per_row * r1, 0.0)
    rows = int((target_s - fixed) / per_row)
    rows = min(A.shape[0], max(r2, (rows // threads) * threads))
    v, dt = oracle_rows_tflops(A, B, rows, threads)
    return rows, v, dt, per_row, fixed


def cpu_model() -> str:
    """The host CPU's model name (lscpu's "Model name", else /proc/cpuinfo's), with its vendor."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10, env=dict(os.environ, LC_ALL="C"))
        fields = dict(line.split(":", 1) for line in out.stdout.splitlines() if ":" in line)
        fields = {k.strip(): v.strip() for k, v in fields.items()}
        name = fields.get("Model name")
        if name:
            vendor = fields.get("Vendor ID")
            return f"{vendor} {name}" if vendor and vendor not in name else name
    except (OSError, subprocess.SubprocessError, ValueError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


def cpu_baseline(A, B, target_s: float = 12.0) -> dict:
    threads = os.cpu_count() or 1
    rows, v, dt, _, _ = oracle_rows_calibrated(A, B, threads, target_s)
    return {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"rows 0..{rows - 1} of D for {WORKLOAD} ({rows}x{B.shape[0]} outputs, K={A.shape[1]}), "
                      f"{dt:.1f} s on {threads} host threads"}


def oracle_workload_timing(w, A, B, target_s: float = 1.5) -> dict:
    """The oracle as it stands on one workload, in seconds and GFLOP/s: one host thread on the
    whole product for the two small shapes, all host threads on a bounded number of full rows of
    D for the large ones (then also the full product's time, scaled from the rows)."""
    import oracle

    small = w.flop < 1e9
    threads = 1 if small else (os.cpu_count() or 1)
    if small:
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.gemm_f16_nt(A, B, threads=1)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= 0.2:
                break
        per = dt / reps
        return {"threads": 1, "seconds": per, "gflops": w.flop / per / 1e9,
                "sample": f"the whole product, {reps} calls"}
    rows, tf, dt, _, _ = oracle_rows_calibrated(A, B, threads, target_s)
    return {"threads": threads, "seconds": dt, "gflops": tf * 1e3, "full_product_seconds": dt * w.M / rows,
            "sample": f"rows 0..{rows - 1} of D ({rows} of {w.M}); the full product's time scaled linearly "
                      f"from the sample"}


def run_reference(args) -> None:
    """--impl reference: the oracle timed on the host cores, each step a bounded sample."""
    import oracle

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = si.WORKLOADS[WORKLOAD]
    A, B = w.operands()
    threads = os.cpu_count() or 1
    oracle.build()
    # size each step so that warm-up + timed steps take about --ref-seconds (a minute) in total
    rng = np.random.default_rng(0)
    calib = 2048
    t0 = time.perf_counter()
    oracle.gemm_f16_nt_points(A, B, rng.integers(0, w.M, calib), rng.integers(0, w.N, calib), threads=threads)
    per_point = (time.perf_counter() - t0) / calib
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    points = int(min(1 << 20, max(threads, budget / per_point)))
    samples = [(rng.integers(0, w.M, points), rng.integers(0, w.N, points)) for _ in range(2)]
    for i in range(args.warmup):
        oracle.gemm_f16_nt_points(A, B, *samples[i % 2], threads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.gemm_f16_nt_points(A, B, *samples[i % 2], threads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * points * w.K * args.steps
    value = flops / dt / 1e12
    sample = f"{points} random output points of {WORKLOAD} per step (K={w.K} each), oracle on {threads} host threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": w.M, "N": w.N, "K": w.K, "seed": w.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------ all five workloads --

def measure_all_workloads(g, dev, peak: float, A3=None, B3=None, budget_s: float = 0.4,
                          oracle_timing: bool = False) -> list[dict]:
    """Each synthetic shape once: TFLOP/s, fraction of the tensor peak, and HBM GB/s of the
    compulsory bytes (the figure that matters for the small, latency-bound shapes).
    With `oracle_timing` (the cpu_baseline leg) sampled outputs of each shape are checked
    against the oracle and the oracle is timed on each shape; without it the oracle is not run.

    Inputs rotate over enough device copies that one pass through them exceeds
    the 129 MB L2 (one copy when a single problem already does), so every
    launch reads A and B from HBM.  The launches are captured once in a CUDA
    graph and the graph is replayed, so the small shapes are timed on the
    device, not by the host's launch rate.  cuBLAS (torch.matmul) runs the
    same way on the same rotation as a reference point.
    """
    import torch

    if oracle_timing:
        import oracle

    torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = False
    out = []
    stream = torch.cuda.Stream(dev)
    for name in si.WORKLOAD_ORDER:
        w = si.WORKLOADS[name]
        A, B = (A3, B3) if (name == si.HEADLINE and A3 is not None) else w.operands()
        rot = 1 if w.min_bytes > (256 << 20) else min(4096, -(-(256 << 20) // w.min_bytes))
        with torch.cuda.stream(stream):
            Ar = torch.from_numpy(A).to(dev).unsqueeze(0).repeat(rot, 1, 1)
            Br = torch.from_numpy(B).to(dev).unsqueeze(0).repeat(rot, 1, 1)
            Dr = torch.empty((rot, w.M, w.N), dtype=torch.float16, device=dev)
        stream.synchronize()
        sh = stream.cuda_stream

        def ours(i):
            j = i % rot
            rc = g.gemm_f16_nt_ptr(Ar[j].data_ptr(), Br[j].data_ptr(), Dr[j].data_ptr(), w.M, w.N, w.K, sh)
            if rc != 0:
                raise g.GemmError(rc, f"gemm_f16_nt ({name})")

        def cublas(i):
            j = i % rot
            with torch.cuda.stream(stream):
                torch.matmul(Ar[j], Br[j].t(), out=Dr[j])

        ours(0)
        if g.last_device_status(stream)[0] != 0:
            raise RuntimeError(f"device status after {name}")
        parity = None
        if oracle_timing:
            rng = np.random.default_rng(7)
            pr, pc = rng.integers(0, w.M, 256), rng.integers(0, w.N, 256)
            ref = oracle.gemm_f16_nt_points(A, B, pr, pc).view(np.float16).astype(np.float64)
            got = Dr[0].cpu().numpy()[pr, pc].astype(np.float64)
            parity = parity_stats(got, ref)
            if not parity["pass"]:
                raise RuntimeError(f"correctness guard failed for {name}")
        replays = 10
        per_graph = int(min(400, max(10, budget_s / replays / max(w.flop / 1.5e15, 3e-6))))
        cfg = g.describe(w.M, w.N, w.K)
        res = {"workload": name, "M": w.M, "N": w.N, "K": w.K, "steps": per_graph * replays,
               "kernel": {k: cfg[k] for k in ("cta_group", "consumers", "block_n", "block_m", "split_k", "cluster_k",
                                              "clusters", "work_items")},
               "parity_vs_oracle": parity,
               "rotated_copies": rot,
               "timing": f"CUDA graph of {per_graph} launches, replayed {replays} times; "
                         "percentiles over the per-replay mean"}
        for label, fn in (("ours", ours), ("cublas", cublas)):
            for i in range(5):
                fn(i)
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                for i in range(per_graph):
                    fn(i)
            # one event per replay boundary: the spread over replays gives p10 / median / p90
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
            with torch.cuda.stream(stream):
                graph.replay()  # warm-up replay
                ev[0].record(stream)
                for r in range(replays):
                    graph.replay()
                    ev[r + 1].record(stream)
            ev[-1].synchronize()
            del graph
            per = sorted(ev[r].elapsed_time(ev[r + 1]) / per_graph for r in range(replays))
            ms = ev[0].elapsed_time(ev[-1]) / (per_graph * replays)
            tf = w.flop / (ms * 1e-3) / 1e12
            pct = {"ms_p10": float(np.percentile(per, 10)), "ms_median": float(np.percentile(per, 50)),
                   "ms_p90": float(np.percentile(per, 90))}
            if label == "ours":
                res.update(ms_per_step=ms, tflops=tf, frac_of_peak=tf / peak,
                           hbm_gbs_compulsory=w.min_bytes / (ms * 1e-3) / 1e9, **pct)
            else:
                res["cublas_tflops"] = tf
                res["cublas_ms_median"] = pct["ms_median"]
        if oracle_timing:
            res["oracle"] = oracle_workload_timing(w, A, B)
        out.append(res)
        del Ar, Br, Dr
        torch.cuda.empty_cache()
    return out


# --------------------------------------------------- sustained, at the cap --

def measure_sustained(g, dev, A, B, local: int, seconds: float, with_cublas: bool = True) -> dict:
    """The headline GEMM back to back for `seconds` per window, ours and cuBLAS alternating
    (ours, cuBLAS, ours, cuBLAS), each window a CUDA graph of launches replayed over and over
    with the inputs rotating over ROTATE device copies, its SM clock sampled inside the window.
    Long windows run at the power cap, where the clock follows the power; the fraction of the
    measured sustained peak (a cuBLAS bf16 loop under the same cap) is the fair comparison."""
    import torch

    w = si.WORKLOADS[WORKLOAD]
    flop = float(w.flop)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    with torch.cuda.stream(stream):
        a0, b0 = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
        As = [a0.clone() for _ in range(ROTATE)]
        Bs = [b0.clone() for _ in range(ROTATE)]
        Ds = [torch.empty((w.M, w.N), dtype=torch.float16, device=dev) for _ in range(ROTATE)]
        del a0, b0
    stream.synchronize()
    torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = False

    def ours(i):
        j = i % ROTATE
        rc = g.gemm_f16_nt_ptr(As[j].data_ptr(), Bs[j].data_ptr(), Ds[j].data_ptr(), w.M, w.N, w.K, sh)
        if rc != 0:
            raise g.GemmError(rc, "gemm_f16_nt (sustained)")

    def cublas(i):
        j = i % ROTATE
        torch.matmul(As[j], Bs[j].t(), out=Ds[j])

    per_graph = 100
    graphs = {}
    for label, fn in (("ours", ours), ("cublas", cublas)):
        if label == "cublas" and not with_cublas:
            continue
        with torch.cuda.stream(stream):
            for i in range(5):
                fn(i)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for i in range(per_graph):
                fn(i)
        graphs[label] = graph
    windows = {label: [] for label in graphs}
    for label in list(graphs) * 2:
        graph = graphs[label]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            graph.replay()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        e1.synchronize()
        replays = max(1, int(seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
        sampler = ClockSampler(local, interval_ms=20.0)
        sampler.wait_for_sample(0.0)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(replays):
                graph.replay()
            ev1.record(stream)
        ev1.synchronize()
        t1 = time.time()
        clocks = sampler.summary(t0, t1)
        sampler.stop()
        ms = ev0.elapsed_time(ev1) / (replays * per_graph)
        tf = flop / (ms * 1e-3) / 1e12
        win = {"tflops": tf, "us_per_gemm": ms * 1e3, "gemms": replays * per_graph,
               "seconds": ev0.elapsed_time(ev1) * 1e-3, "sm_mhz": clocks.get("sm_mhz"),
               "reasons": clocks.get("reasons"), "power_w_max": clocks.get("power_w_max"),
               "samples": clocks.get("samples")}
        if clocks.get("sm_mhz"):
            win["tflops_per_ghz"] = tf / (clocks["sm_mhz"] / 1000.0)
        windows[label].append(win)
    status, info = g.last_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {g.status_string(status)} info={info:#x}")
    del graphs, As, Bs, Ds
    torch.cuda.empty_cache()

    def mean(label, key):
        vals = [x[key] for x in windows[label] if x.get(key) is not None]
        return statistics.fmean(vals) if vals else None

    ours_tf = mean("ours", "tflops")
    out = {"value": ours_tf, "unit": UNIT, "sm_mhz": mean("ours", "sm_mhz"),
           "tflops_per_ghz": mean("ours", "tflops_per_ghz"), "windows": windows["ours"]}
    if "cublas" in windows:
        cb = mean("cublas", "tflops")
        out["cublas"] = {"value": cb, "sm_mhz": mean("cublas", "sm_mhz"),
                         "tflops_per_ghz": mean("cublas", "tflops_per_ghz"), "windows": windows["cublas"]}
        out["vs_cublas"] = ours_tf / cb if cb else None
    out["what"] = (f"{WORKLOAD} back to back, CUDA-graph replay, {seconds:g} s windows alternating ours / cuBLAS "
                   f"twice; value = mean of our two windows; clocks sampled inside each window")
    return out


def kernel_label(cfg: dict) -> str:
    """A short name for the configuration gemm_f16_nt_describe reports."""
    if cfg["block_n"] == 16:
        kind = "thin 64x16"
    elif cfg["block_n"] == 64:
        kind = f"{'tiny' if cfg['block_m'] == 64 else 'narrow'} {cfg['block_m']}x64"
        if cfg["cluster_k"] > 1:
            kind += f", K over {cfg['cluster_k']} CTAs"
    else:
        kind = ("pair" if cfg["cta_group"] == 2 else "single") + f" {128 * cfg['cta_group'] * cfg['consumers']}x256"
        if cfg["consumers"] == 2:
            kind += ", 2 consumers"
    return f"{kind}, {cfg['clusters']} clusters"


def workloads_summary(workloads: list[dict]) -> list[dict]:
    """One short entry per workload (graph-timed median), for the end of the JSON line."""
    out = []
    for w in workloads:
        p = w.get("parity_vs_oracle")
        out.append({"workload": w["workload"], "kernel": kernel_label(w["kernel"]),
                    "us": round(w["ms_median"] * 1e3, 2), "tflops": round(w["tflops"], 1),
                    "cublas_us": round(w["cublas_ms_median"] * 1e3, 2) if w.get("cublas_ms_median") else None,
                    "hbm_gbs": round(w["hbm_gbs_compulsory"], 1), "parity": p["pass"] if p else None})
    return out


# ---------------------------------------------------------------- GPU arm --

def run_ours(args) -> None:
    import torch

    import blackwell_tensor_core_02_gb300 as g

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    g.load()
    w = si.WORKLOADS[WORKLOAD]
    A, B = w.operands()
    flop = float(w.flop)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    As, Bs, Ds = [], [], []
    with torch.cuda.stream(stream):
        a0 = torch.from_numpy(A).to(dev)
        b0 = torch.from_numpy(B).to(dev)
        for _ in range(ROTATE):
            As.append(a0.clone())
            Bs.append(b0.clone())
            Ds.append(torch.empty((w.M, w.N), dtype=torch.float16, device=dev))
        del a0, b0
    stream.synchronize()

    def step(i):
        j = i % ROTATE
        rc = g.gemm_f16_nt_ptr(As[j].data_ptr(), Bs[j].data_ptr(), Ds[j].data_ptr(), w.M, w.N, w.K, sh)
        if rc != 0:
            raise g.GemmError(rc, "gemm_f16_nt")

    step(0)
    status, info = g.last_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {g.status_string(status)} info={info:#x}")
    # the cpu_baseline leg (rank 0 of one GPU), before anything is timed: the oracle on a few
    # sampled outputs of the timed configuration, a guard that stops the run on a mismatch
    cpu_leg = rank == 0 and world == 1 and not args.no_cpu_baseline
    parity = None
    if cpu_leg:
        import oracle

        rng = np.random.default_rng(1)
        pr, pc = rng.integers(0, w.M, 512), rng.integers(0, w.N, 512)
        ref = oracle.gemm_f16_nt_points(A, B, pr, pc).view(np.float16).astype(np.float64)
        got = Ds[0].cpu().numpy()[pr, pc].astype(np.float64)
        parity = parity_stats(got, ref)
        if not parity["pass"]:
            raise RuntimeError("bench correctness guard failed against the oracle")

    def timed_region():
        """W warm-up steps, then K timed steps between barriers; (max elapsed ms over ranks,
        rank 0's clock record of the timed region)."""
        sampler = ClockSampler(local) if rank == 0 else None
        if sampler:
            sampler.wait_for_sample(0.0)  # nvidia-smi is up and sampling before anything is timed
        for i in range(args.warmup):
            step(i)
        barrier()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        t_wall0 = time.time()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        ev1.synchronize()
        t_wall1 = time.time()
        barrier()
        ms = ev0.elapsed_time(ev1)
        status, info = g.last_device_status(stream)
        if status != 0:
            raise RuntimeError(f"device status {g.status_string(status)} info={info:#x}")
        ms = max_over_ranks(ms, dist, dev)
        record = sampler.summary(t_wall0, t_wall1) if sampler else None
        if sampler:
            sampler.stop()
        return ms, record

    elapsed_ms, clocks = timed_region()
    # a run the clock record disqualifies is measured once more (every rank, in step)
    if max_over_ranks(1.0 if needs_remeasure(clocks) else 0.0, dist, dev) > 0:
        first = clocks
        elapsed_ms, clocks = timed_region()
        if clocks is not None:
            clocks["remeasured_after"] = {k: first.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")} if first else None

    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tflops(flop, args.steps, world, elapsed_ms)
    per_gpu_tflops = flop / (ms_per_step * 1e-3) / 1e12
    if clocks and clocks.get("sm_mhz"):
        # under the power cap the clock follows the power: the work done per clock is what
        # the kernel decides (nvidia-smi's power reading averages over about a second, too
        # long for a per-joule figure over this timed region)
        clocks["tflops_per_ghz"] = per_gpu_tflops / (clocks["sm_mhz"] / 1000.0)

    # cuBLAS (torch.matmul) on the same rotation, as a reference point
    cublas = None
    if not args.no_cublas:
        torch.backends.cuda.matmul.allow_fp16_reduced_precision_reduction = False
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                torch.matmul(As[i % ROTATE], Bs[i % ROTATE].t(), out=Ds[i % ROTATE])
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for i in range(args.steps):
                torch.matmul(As[i % ROTATE], Bs[i % ROTATE].t(), out=Ds[i % ROTATE])
            c1.record(stream)
        c1.synchronize()
        cms = c0.elapsed_time(c1) / args.steps
        cublas = {"value": flop / (cms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": cms,
                  "what": "torch.matmul(A, B.T) (cuBLAS), fp16 reduced-precision reduction off, same rotation"}

    # end to end through the public host-buffer API: every step copies its A
    # and B in from pinned host memory, runs the GEMM and copies D back out;
    # HostPipeline overlaps step i's GEMM with step i+1's copy-in and step
    # i-1's copy-out on separate streams
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(B).pin_memory()
    Dh = [torch.empty((w.M, w.N), dtype=torch.float16).pin_memory() for _ in range(2)]
    del As, Bs, Ds
    pipe = g.HostPipeline(w.M, w.N, w.K, device=dev)
    for i in range(min(3, args.warmup)):
        pipe.submit(Ah, Bh, Dh[i % 2])
    pipe.synchronize()
    barrier()
    t_e0 = time.perf_counter()
    e0 = pipe.record_start()
    for i in range(e2e_steps):
        pipe.submit(Ah, Bh, Dh[i % 2])
    e1 = pipe.record_end()
    pipe.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_wall_ms = (time.perf_counter() - t_e0) * 1e3
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = whole_job_tflops(flop, e2e_steps, world, e2e_ms)

    if rank == 0:
        peak, peak_sustained, peak_src = measured_peak()
        roof_peak, regime, roof_src = roofline_peak(elapsed_ms / 1e3, peak, peak_sustained, peak_src)
        traffic, traffic_src = ncu_traffic()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": w.M, "N": w.N, "K": w.K, "seed": w.seed,
                       "inputs": "fp16 uniform[-1,1], splitmix64 seed 2; fp32 accumulation, fp16 output",
                       "l2": f"inputs larger than L2: A, B, D rotate over {ROTATE} device copies "
                             f"({ROTATE * w.min_bytes / 2 ** 20:.0f} MiB)",
                       "cta_group": 2, "tile": "256x256 per CTA pair", "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": per_gpu_tflops, "peak": roof_peak, "unit": UNIT,
                         "frac": per_gpu_tflops / roof_peak, "traffic": traffic, "kernel": KERNEL_NAME,
                         "peak_source": roof_src, "peak_regime": regime,
                         "frac_of_burst": per_gpu_tflops / peak,
                         "frac_of_sustained": (per_gpu_tflops / peak_sustained) if peak_sustained else None,
                         "stated_peak": STATED_PEAK_TFLOPS,
                         "frac_of_stated_peak": per_gpu_tflops / STATED_PEAK_TFLOPS,
                         "traffic_source": traffic_src,
                         "algorithmic_flop_per_launch": flop,
                         "algorithmic_bytes_per_launch": w.min_bytes},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 2 * (w.M * w.K + w.N * w.K),
                    "d2h_bytes_per_step": 2 * w.M * w.N, "steps": e2e_steps, "wall_ms": e2e_wall_ms,
                    "what": "HostPipeline: per step one gemm_f16_nt_host call (C ABI: pinned host A, B -> "
                            "device, GEMM, D -> pinned host, enqueued on one stream); three slots on three "
                            "streams overlap neighbouring steps' copies with the GEMM"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cublas_reference": cublas,
            "parity_vs_oracle": parity,
        }
        if cpu_leg:
            line["cpu_baseline"] = cpu_baseline(A, B)
        if world == 1 and not args.no_workloads:
            line["workloads"] = measure_all_workloads(g, dev, peak, A, B, oracle_timing=cpu_leg)
        if world == 1 and args.sustained_seconds > 0:
            sus = measure_sustained(g, dev, A, B, local, args.sustained_seconds, with_cublas=not args.no_cublas)
            if peak_sustained:
                sus["frac_of_measured_sustained"] = sus["value"] / peak_sustained
            sus["frac_of_stated_peak"] = sus["value"] / STATED_PEAK_TFLOPS
            line["sustained"] = sus
        if "workloads" in line:
            # last, so that a reader of the line's tail sees all five shapes
            line["workloads_summary"] = workloads_summary(line["workloads"])
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the pass over all five shapes")
    ap.add_argument("--sustained-seconds", type=float, default=2.0,
                    help="length of each back-to-back window of the sustained (power-capped) measurement; 0: none")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: host time for warm-up and timed steps together")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if not args.ref_seconds > 0:
        ap.error("--ref-seconds must be positive")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
