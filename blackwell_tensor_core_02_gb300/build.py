"""Build the sm_103a CUDA library in-tree (nvcc, one translation unit).

The result is ``blackwell_tensor_core_02_gb300/_build/libgemm_f16.so``; it
exports exactly the C ABI declared in ``include/gemm_f16.h``.  A second build
of the same source with the device range checks compiled in
(``-DGEMM_F16_DEVICE_CHECKS=1``), ``libgemm_f16_checked.so``, is for tests.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libgemm_f16.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
CHECKED_LIB_PATH = os.path.join(BUILD_DIR, "libgemm_f16_checked.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the sm_103a library cannot be built")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(INCLUDE, "gemm_f16.h")])


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    built = os.path.getmtime(path)
    return any(os.path.getmtime(s) > built for s in sources())


def _command(path: str, checked: bool, verbose: bool) -> list[str]:
    return [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            *(["-DGEMM_F16_DEVICE_CHECKS=1"] if checked else []), *(["-Xptxas", "-v"] if verbose else []),
            "-I", INCLUDE, "-I", CSRC, os.path.join(CSRC, "gemm_f16.cu"), "-o", path]


def build_many(targets: list[tuple[str, bool]], force: bool = False, verbose: bool = False) -> None:
    """Compile the (path, checked) targets that are missing or stale, in parallel."""
    todo = [(path, checked) for path, checked in targets if force or is_stale(path)]
    if not todo:
        return
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    for path, checked in todo:
        tmp = f"{path}.{os.getpid()}.tmp"
        cmd = _command(tmp, checked, verbose)
        procs.append((path, tmp, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
    errors = []
    for path, tmp, cmd, proc in procs:
        out, err = proc.communicate()
        if proc.returncode != 0:
            errors.append(f"nvcc failed ({proc.returncode}):\n{' '.join(cmd)}\n{out}\n{err}")
            continue
        if verbose:
            print(out + err)
        os.replace(tmp, path)
    if errors:
        raise RuntimeError("\n".join(errors))


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile the library (or its checked build) if missing or older than its sources; return its path."""
    path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_many([(path, checked)], force=force, verbose=verbose)
    return path


def build_all(force: bool = False, verbose: bool = False) -> None:
    """Both builds, compiled side by side."""
    build_many([(LIB_PATH, False), (CHECKED_LIB_PATH, True)], force=force, verbose=verbose)


if __name__ == "__main__":
    build_all(force=True, verbose=True)
    print(LIB_PATH)
    print(CHECKED_LIB_PATH)
