"""Host logic of bench.py: the cross-rank reduction (2 gloo ranks on CPU) and the CLI contract."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [10.0, 12.5][rank]  # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed, dist, "cpu")
    v = bench.whole_job_tflops(1e12, 100, world, m)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": m, "value": v}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks(tmp_path):
    torch = pytest.importorskip("torch")
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.multiprocessing.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert res[0] == res[1]
    assert res[0]["max"] == 12.5
    # 2 replicas x 100 steps x 1 TFLOP in 12.5 ms
    assert res[0]["value"] == pytest.approx(2 * 100 * 1e12 / 12.5e-3 / 1e12)


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_tflops(2e12, 10, 1, 20.0) == pytest.approx(1000.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_clock_records_that_disqualify_a_run():
    # kept: the power cap of a dense GEMM, and clocks near the maximum
    assert not bench.needs_remeasure({"sm_mhz": 1520.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    assert not bench.needs_remeasure({"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert not bench.needs_remeasure(None)
    assert not bench.needs_remeasure({"sm_mhz": None, "sm_max_mhz": None, "reasons": []})
    # measured again: a hardware or thermal slowdown, or clocks far down with no reason (a lock)
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.needs_remeasure({"sm_mhz": 1400.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap", r]})
    assert bench.needs_remeasure({"sm_mhz": 1000.0, "sm_max_mhz": 2070.0, "reasons": []})


def test_reference_arm_prints_the_contract_line():
    """--impl reference on the host cores: one JSON line with the main arm's metric, unit and
    direction, the oracle as its cpu_baseline, and an e2e that moves no bytes to or from a GPU."""
    env = dict(os.environ, RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "3", "--ref-seconds", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert (d["impl"], d["metric"], d["unit"], d["higher_is_better"]) == ("reference", bench.METRIC, bench.UNIT, True)
    assert (d["n_gpus"], d["steps"], d["warmup"], d["data"], d["dtype"]) == (1, 2, 3, "synthetic", "f64")
    assert d["config"]["workload"] == bench.WORKLOAD and d["value"] > 0 and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_budget_must_be_positive():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--ref-seconds", "0"],
                         cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert out.returncode != 0 and "--ref-seconds" in out.stderr


def test_roofline_peak_follows_the_length_of_the_timed_region():
    """A long back-to-back region runs under the power cap and is set against the measured
    sustained peak; a short burst against the burst peak; with no sustained figure, burst."""
    peak, regime, src = bench.roofline_peak(0.86, 1912.4, 1724.7, "burst source")
    assert (peak, regime) == (1724.7, "sustained") and "sustained" in src and "0.86 s" in src
    assert bench.roofline_peak(0.0017, 1912.4, 1724.7, "burst source") == (1912.4, "burst", "burst source")
    assert bench.roofline_peak(5.0, 1912.4, None, "burst source") == (1912.4, "burst", "burst source")
    assert bench.roofline_peak(bench.SUSTAINED_REGION_S, 1912.4, 1724.7, "b")[1] == "sustained"



def test_kernel_labels_name_each_configuration():
    """The compact workload list names the kernel from gemm_f16_nt_describe's fields."""
    base = dict(cta_group=1, consumers=1, block_n=64, block_m=64, cluster_k=1, clusters=16)
    assert bench.kernel_label({**base, "block_n": 16}) == "thin 64x16, 16 clusters"
    assert bench.kernel_label(base) == "tiny 64x64, 16 clusters"
    assert bench.kernel_label({**base, "cluster_k": 4}) == "tiny 64x64, K over 4 CTAs, 16 clusters"
    assert bench.kernel_label({**base, "block_m": 128, "cluster_k": 2}) == "narrow 128x64, K over 2 CTAs, 16 clusters"
    pair = dict(cta_group=2, consumers=1, block_n=256, block_m=128, cluster_k=1, clusters=76)
    assert bench.kernel_label(pair) == "pair 256x256, 76 clusters"
    assert bench.kernel_label({**pair, "consumers": 2}) == "pair 512x256, 2 consumers, 76 clusters"
    assert bench.kernel_label({**pair, "cta_group": 1, "clusters": 152}) == "single 128x256, 152 clusters"


def test_workloads_summary_keeps_one_short_entry_per_workload():
    w = {"workload": "square_4096", "ms_median": 0.0812345, "tflops": 1692.04, "cublas_ms_median": 0.0833,
         "hbm_gbs_compulsory": 1239.11, "parity_vs_oracle": {"pass": True},
         "kernel": dict(cta_group=2, consumers=1, block_n=256, block_m=128, cluster_k=1, clusters=76)}
    [s] = bench.workloads_summary([w])
    assert s == {"workload": "square_4096", "kernel": "pair 256x256, 76 clusters", "us": 81.23, "tflops": 1692.0,
                 "cublas_us": 83.3, "hbm_gbs": 1239.1, "parity": True}
    [s] = bench.workloads_summary([{**w, "cublas_ms_median": None, "parity_vs_oracle": None}])
    assert s["cublas_us"] is None and s["parity"] is None
