"""Time the GEMM on one or more shapes from the command line (also a fixed workload to profile).

    python -m blackwell_tensor_core_02_gb300.drive --shape 1024,1024,4096 --entry ws --graph --cublas
    python -m blackwell_tensor_core_02_gb300.drive --shape 1536,1536,1536 2048,2048,2048 --graph --cublas
    python -m blackwell_tensor_core_02_gb300.drive --shape 8192,8192,8192 --consumers 1 2 --graph \
        --seconds 1.2 --reps 2

Operands come from the seeded generator (uniform[-1, 1], seed 1) and rotate
over enough device copies that one pass exceeds the 129 MB L2.  ``--entry``
picks the C entry point: ``nt`` (gemm_f16_nt_ex, no workspace), ``ws``
(gemm_f16_nt_ws with a workspace sized by gemm_f16_nt_workspace_size) or
``static`` (gemm_f16_nt_static_ws).  With ``--graph`` the launches are captured
in a CUDA graph; ``--seconds S`` then replays it back to back for S seconds per
measurement (long enough to reach the power cap) and samples the SM clock
meanwhile.  Several ``--consumers`` values (and cuBLAS with ``--cublas``) are
measured one after the other, ``--reps`` times over.  Prints one JSON line per
measurement.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)


def main(argv=None) -> None:
    import ctypes

    import torch

    import blackwell_tensor_core_02_gb300 as g
    import seeded_inputs as si
    from blackwell_tensor_core_02_gb300.clocks import ClockSampler

    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--shape", required=True, nargs="+", help="M,N,K (several: one after the other)")
    ap.add_argument("--entry", choices=["nt", "ws", "static"], default="nt")
    ap.add_argument("--cta-group", type=int, default=0)
    ap.add_argument("--consumers", type=int, nargs="+", default=[0],
                    help="MMA consumers 1 or 2, 0 for the shape's default; several: each in turn")
    ap.add_argument("--block-n", type=int, default=0, help="tile width: 16 (thin 64 x 16 tiles), 64, 256, or 0 for the shape's default")
    ap.add_argument("--block-m", type=int, default=0, help="rows per CTA: 64 (with 64-wide tiles), 128, or 0")
    ap.add_argument("--cluster-k", type=int, default=0,
                    help="tiny tiles: K split across clusters of 2, 4 or 8 CTAs; 1 none; 0 the shape's default")
    ap.add_argument("--raster-group", type=int, default=0,
                    help="M-tiles per group of the tile order; 0 for the shape's default")
    ap.add_argument("--steps", type=int, default=200, help="launches per timed run (per graph with --graph)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--graph", action="store_true", help="time a CUDA graph of the launches")
    ap.add_argument("--seconds", type=float, default=0.0,
                    help="with --graph: replay the graph back to back for this long per measurement, clocks sampled")
    ap.add_argument("--reps", type=int, default=1, help="measure every variant this many times, alternating")
    ap.add_argument("--cublas", action="store_true", help="also time torch.matmul on the same rotation")
    args = ap.parse_args(argv)
    lib = g.load()
    dev = torch.device("cuda")
    for shape in args.shape:
        M, N, K = (int(x) for x in shape.split(","))
        A, B = si.custom(M, N, K, seed=1).operands()
        footprint = 2 * (M * K + N * K + M * N)
        rot = max(1, min(256, (256 << 20) // max(footprint, 1)))
        Ar = torch.from_numpy(A).to(dev).unsqueeze(0).repeat(rot, 1, 1)
        Br = torch.from_numpy(B).to(dev).unsqueeze(0).repeat(rot, 1, 1)
        Dr = torch.empty((rot, M, N), dtype=torch.float16, device=dev)
        stream = torch.cuda.Stream()
        sh = stream.cuda_stream

        def ours_for(consumers):
            opts = g.Options(cta_group=args.cta_group, consumers=consumers, block_n=args.block_n,
                             block_m=args.block_m, cluster_k=args.cluster_k, raster_group=args.raster_group)
            need = g.workspace_size(M, N, K, opts) if args.entry == "ws" else 0
            ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

            def ours(i):
                j = i % rot
                a, b, d = Ar[j].data_ptr(), Br[j].data_ptr(), Dr[j].data_ptr()
                if args.entry == "ws":
                    rc = g.gemm_f16_nt_ptr(a, b, d, M, N, K, sh, opts, ws.data_ptr(), need)
                elif args.entry == "static":
                    rc = lib.gemm_f16_nt_static_ws(a, b, d, M, N, K, sh, ctypes.byref(opts))
                else:
                    rc = g.gemm_f16_nt_ptr(a, b, d, M, N, K, sh, opts)
                if rc != 0:
                    raise g.GemmError(rc, "drive")

            ours.workspace = need
            ours.config = g.describe(M, N, K, opts, with_workspace=args.entry != "nt")
            return ours

        def cublas(i):
            j = i % rot
            torch.matmul(Ar[j], Br[j].t(), out=Dr[j])

        runs = [("ours", c, ours_for(c)) for c in args.consumers]
        if args.cublas:
            runs.append(("cublas", None, cublas))
        for rep in range(args.reps):
            for label, consumers, fn in runs:
                with torch.cuda.stream(stream):
                    for i in range(args.warmup):
                        fn(i)
                stream.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                clocks = None
                launches = args.steps
                if args.graph:
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                        for i in range(args.steps):
                            fn(i)
                    with torch.cuda.stream(stream):
                        graph.replay()
                        e0.record(stream)
                        graph.replay()
                        e1.record(stream)
                    e1.synchronize()
                    if args.seconds > 0:
                        replays = max(1, int(args.seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
                        sampler = ClockSampler(torch.cuda.current_device(), interval_ms=10.0)
                        sampler.wait_for_sample(0.0)
                        t0 = time.time()
                        with torch.cuda.stream(stream):
                            e0.record(stream)
                            for _ in range(replays):
                                graph.replay()
                            e1.record(stream)
                        e1.synchronize()
                        clocks = sampler.summary(t0, time.time())
                        sampler.stop()
                        launches = args.steps * replays
                    del graph
                else:
                    with torch.cuda.stream(stream):
                        e0.record(stream)
                        for i in range(args.steps):
                            fn(i)
                        e1.record(stream)
                    e1.synchronize()
                us = e0.elapsed_time(e1) / launches * 1e3
                tflops = 2.0 * M * N * K / (us * 1e-6) / 1e12
                status = g.last_device_status(stream)[0]
                out = {"impl": label, "shape": [M, N, K], "rep": rep, "entry": args.entry if label == "ours" else None,
                       "config": fn.config if label == "ours" else None,
                       "workspace_bytes": fn.workspace if label == "ours" else 0, "us_per_gemm": round(us, 3),
                       "tflops": round(tflops, 2), "graph": args.graph, "status": status}
                if clocks is not None:
                    out.update(seconds=round(e0.elapsed_time(e1) * 1e-3, 3), sm_mhz=clocks.get("sm_mhz"),
                               reasons=clocks.get("reasons"),
                               tflops_per_ghz=round(tflops / (clocks["sm_mhz"] / 1000.0), 1)
                               if clocks.get("sm_mhz") else None)
                print(json.dumps(out), flush=True)
        del Ar, Br, Dr
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
