"""Compile-time facts of the sm_103a kernels, read from ptxas's own report (-Xptxas -v; no GPU).

* No kernel instantiation spills registers or keeps a stack frame.
* The two-consumer kernel launches 384 threads with exactly 168 registers each: its
  register split ("GEMM III -- warp specialization & clusters to SOTA", Step 7, setmaxnreg)
  moves warpgroup 0 down to 40 and the two epilogue warpgroups up to 232, which adds up to
  384 x 168 = 64 512, the whole pool the CTA launches with.  With fewer registers per thread at
  launch an increase would wait for registers that never come; the library also refuses to run
  if the loaded kernel reports another count.
"""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "blackwell_tensor_core_02_gb300", "csrc")


@pytest.fixture(scope="module")
def ptxas_report(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = tmp_path_factory.mktemp("regs") / "gemm.cubin"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-cubin",
                        "-Xptxas", "-v", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                        os.path.join(CSRC, "gemm_f16.cu"), "-o", str(out)], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    kernels = {}
    current = None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            current = m.group(1)
            kernels[current] = {}
            continue
        if current is None:
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            kernels[current].update(stack=int(m.group(1)), spill_st=int(m.group(2)), spill_ld=int(m.group(3)))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            kernels[current]["regs"] = int(m.group(1))
    return kernels


def _gemm_kernels(report):
    out = {}
    for name, info in report.items():
        m = re.search(r"gemm_f16_nt_kernelILi(\d+)ELi(\d+)ELi(\d+)ELi(\d+)ELi(\d+)E", name)
        if m:
            out[tuple(int(x) for x in m.groups())] = info
    return out


def test_no_kernel_spills(ptxas_report):
    assert len(_gemm_kernels(ptxas_report)) >= 11
    for name, info in ptxas_report.items():
        assert info.get("spill_st") == 0 and info.get("spill_ld") == 0 and info.get("stack") == 0, (name, info)


def test_two_consumer_kernel_launches_with_the_whole_register_pool(ptxas_report):
    k = _gemm_kernels(ptxas_report)
    assert k[(2, 2, 256, 128, 1)]["regs"] == 168  # (65536 / 384) rounded down to a multiple of 8
    assert 128 * 40 + 256 * 232 == 384 * 168
    # every other instantiation stays within what one CTA per SM allows
    for cfg, info in k.items():
        threads = 384 if cfg[1] == 2 else 192
        assert info["regs"] * threads <= 65536, (cfg, info)
