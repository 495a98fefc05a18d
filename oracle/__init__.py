"""CPU oracle for the fp16 GEMM D = A·Bᵀ (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package. The product path —
the CUDA library under ``blackwell_tensor_core_02_gb300`` — never does, and the
oracle shares no code with it.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64 accumulation, one
round-to-nearest-even cast to fp16 at the end; see that file's header for the
passages it follows). This module compiles it with gcc on first use and wraps
it with ctypes. Every function is pinned by ``tests/test_oracle_pins.py``
against the fp16 definition, closed forms, exact brute force and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(mutant: int = 0) -> str:
    name = "libgemm_oracle.so" if mutant == 0 else f"libgemm_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD_DIR, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (``mutant`` > 0 plants a known mistake, for pin tests)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", *_CFLAGS, f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant in _libs:
            return _libs[mutant]
        lib = ctypes.CDLL(build(mutant))
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f16.restype = ctypes.c_uint16
        lib.oracle_f16_to_f64_array.argtypes = [u16p, f64p, i64]
        lib.oracle_f16_to_f64_array.restype = None
        lib.oracle_f64_to_f16_array.argtypes = [f64p, u16p, i64]
        lib.oracle_f64_to_f16_array.restype = None
        lib.oracle_gemm_f16_nt.argtypes = [u16p, u16p, u16p, f64p, i64, i64, i64, ctypes.c_int]
        lib.oracle_gemm_f16_nt.restype = ctypes.c_int
        lib.oracle_gemm_f16_nt_points.argtypes = [u16p, u16p, i64, i64, i64, i64p, i64p, i64, u16p, f64p,
                                                  ctypes.c_int]
        lib.oracle_gemm_f16_nt_points.restype = ctypes.c_int
        _libs[mutant] = lib
        return lib


def _ptr(arr: np.ndarray | None, ctype):
    if arr is None:
        return None
    return arr.ctypes.data_as(ctypes.POINTER(ctype))


def _as_bits(x: np.ndarray) -> np.ndarray:
    """fp16 array (or its uint16 bit pattern) -> contiguous uint16 bits."""
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected float16 or uint16 bits, got {x.dtype}")
    return np.ascontiguousarray(x)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def f16_to_f64(bits: np.ndarray, mutant: int = 0) -> np.ndarray:
    """Decode binary16 bit patterns to doubles (the oracle's own codec)."""
    b = _as_bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load(mutant).oracle_f16_to_f64_array(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double), b.size)
    return out


def f64_to_f16(x: np.ndarray, mutant: int = 0) -> np.ndarray:
    """Round doubles to binary16 bit patterns, ties to even (the oracle's own codec)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    _load(mutant).oracle_f64_to_f16_array(_ptr(x, ctypes.c_double), _ptr(out, ctypes.c_uint16), x.size)
    return out


def gemm_f16_nt(A: np.ndarray, B: np.ndarray, *, with_acc: bool = False, threads: int | None = None,
                mutant: int = 0):
    """D = RNE_fp16(A·Bᵀ) with fp64 accumulation. A is M×K, B is N×K (fp16 or uint16 bits).

    Returns D as uint16 bits (M×N), and with ``with_acc`` also the fp64 sums.
    """
    a, b = _as_bits(A), _as_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch: A {a.shape}, B {b.shape}")
    M, K = a.shape
    N = b.shape[0]
    D = np.empty((M, N), dtype=np.uint16)
    acc = np.empty((M, N), dtype=np.float64) if with_acc else None
    rc = _load(mutant).oracle_gemm_f16_nt(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16),
                                          _ptr(D, ctypes.c_uint16), _ptr(acc, ctypes.c_double), M, N, K,
                                          threads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm_f16_nt failed")
    return (D, acc) if with_acc else D


def gemm_f16_nt_points(A: np.ndarray, B: np.ndarray, rows, cols, *, with_acc: bool = False,
                       threads: int | None = None, mutant: int = 0):
    """The same definition at output points (rows[i], cols[i]); returns uint16 bits [count]."""
    a, b = _as_bits(A), _as_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch: A {a.shape}, B {b.shape}")
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if r.shape != c.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    out = np.empty(r.shape, dtype=np.uint16)
    acc = np.empty(r.shape, dtype=np.float64) if with_acc else None
    rc = _load(mutant).oracle_gemm_f16_nt_points(_ptr(a, ctypes.c_uint16), _ptr(b, ctypes.c_uint16), M, N, K,
                                                 _ptr(r, ctypes.c_int64), _ptr(c, ctypes.c_int64), r.size,
                                                 _ptr(out, ctypes.c_uint16), _ptr(acc, ctypes.c_double),
                                                 threads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm_f16_nt_points failed (index out of range?)")
    return (out, acc) if with_acc else out
