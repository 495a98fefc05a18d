"""Seeded synthetic inputs for the fp16 GEMM D = A·Bᵀ (A M×K, B N×K).

This module holds no GEMM arithmetic. It only draws operands, and both the CUDA
path and the CPU oracle receive the same arrays from it.

Generator (counter based, so any slice can be drawn on its own):
  * splitmix64 (S. Vigna's published finaliser): output i of stream `seed` is
    mix(seed + (i+1)·0x9E3779B97F4A7C15) with the usual two xor-shift-multiply
    rounds;
  * u = (x >> 11)·2⁻⁵³ in [0, 1);
  * uniform[lo, hi): lo + (hi − lo)·u;
  * normal(μ, σ): Box–Muller on consecutive pairs (u₁, u₂):
    r = sqrt(−2·ln(1 − u₁)), z₀ = r·cos(2πu₂), z₁ = r·sin(2πu₂);
  * every value is rounded to fp16 with round-to-nearest-even.
A is drawn first (counters 0 … M·K−1, row-major), then B (counters M·K …).

The five workloads are the synthetic shapes the fp16 GEMM is measured on: a
single 128×128 tile with K=64, a 2×2 grid of tiles with a K-loop, the square
4096³ headline shape, a large 8192³ square, and a transformer MLP projection
(8192 tokens × 28672 × 4096).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start … start+count−1 of the splitmix64 stream seeded with `seed`."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def unit_uniform(seed: int, start: int, count: int) -> np.ndarray:
    """u in [0, 1) with 53 random bits, from counters start … start+count−1."""
    return (splitmix64(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


@dataclass(frozen=True)
class Dist:
    kind: str          # "uniform" or "normal"
    p0: float          # lo, or mean
    p1: float          # hi, or standard deviation

    def draw_f64(self, seed: int, start: int, count: int) -> np.ndarray:
        if self.kind == "uniform":
            return self.p0 + (self.p1 - self.p0) * unit_uniform(seed, start, count)
        if self.kind == "normal":
            if start % 2 or count % 2:
                raise ValueError("normal draws come in pairs: start and count must be even")
            u = unit_uniform(seed, start, count).reshape(-1, 2)
            r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
            t = 2.0 * math.pi * u[:, 1]
            z = np.empty((u.shape[0], 2), dtype=np.float64)
            z[:, 0] = r * np.cos(t)
            z[:, 1] = r * np.sin(t)
            return self.p0 + self.p1 * z.reshape(-1)
        raise ValueError(f"unknown distribution {self.kind}")


def draw_f16(dist: Dist, seed: int, start: int, count: int) -> np.ndarray:
    """`count` fp16 values (RNE) from counters start …; drawn in chunks to bound memory."""
    out = np.empty(count, dtype=np.float16)
    step = _CHUNK
    for off in range(0, count, step):
        n = min(step, count - off)
        if dist.kind == "normal" and n % 2:
            raise ValueError("normal draws need an even element count")
        out[off:off + n] = dist.draw_f64(seed, start + off, n).astype(np.float16)
    return out


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    a: Dist
    b: Dist
    note: str

    @property
    def flop(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """Compulsory fp16 traffic: read A and B once, write D once."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)

    def operands(self) -> tuple[np.ndarray, np.ndarray]:
        """(A, B) as fp16 numpy arrays, A M×K and B N×K, row-major."""
        A = draw_f16(self.a, self.seed, 0, self.M * self.K).reshape(self.M, self.K)
        B = draw_f16(self.b, self.seed, self.M * self.K, self.N * self.K).reshape(self.N, self.K)
        return A, B


_U = Dist("uniform", -1.0, 1.0)

WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("single_tile_128x128x64", 128, 128, 64, 0, _U, _U,
                 "one 128×128 output tile, one 64-wide K chunk"),
        Workload("ktile_grid_256x256x512", 256, 256, 512, 1, _U, _U,
                 "2×2 grid of 128×128 tiles, eight 64-wide K chunks"),
        Workload("square_4096", 4096, 4096, 4096, 2, _U, _U,
                 "square headline shape"),
        Workload("square_8192", 8192, 8192, 8192, 3,
                 Dist("normal", 0.0, 1.0 / math.sqrt(8192)), Dist("normal", 0.0, 1.0 / math.sqrt(8192)),
                 "large square, operands normal(0, 1/sqrt(K))"),
        Workload("mlp_proj_8192x28672x4096", 8192, 28672, 4096, 4,
                 Dist("normal", 0.0, 1.0), Dist("normal", 0.0, 0.02),
                 "transformer MLP projection: activations normal(0,1), weights normal(0,0.02)"),
    ]
}

WORKLOAD_ORDER = list(WORKLOADS)
HEADLINE = "square_4096"


def custom(M: int, N: int, K: int, seed: int, dist: Dist = _U) -> Workload:
    """An ad-hoc workload of the same recipe (for ragged and edge-case shapes)."""
    return Workload(f"custom_{M}x{N}x{K}_s{seed}", M, N, K, seed, dist, dist, "ad hoc")
