"""Pins for the CPU oracle, none of which re-types its formula or re-calls its code.

Each pin rests on something outside the oracle:
  * the IEEE binary16 definition, through numpy's own float16 conversions
    (a library routine) and an exhaustive table of every finite fp16 value;
  * exact rational arithmetic (``fractions.Fraction``) for brute-force sums on
    tiny inputs, rounded once by a nearest-value search over that table;
  * closed forms: identity operands, all-ones (D = K), rank-1 outer products;
  * invariants: swapping A and B transposes D, negating A negates D.

``test_planted_mistakes_are_caught`` rebuilds the oracle with a known mistake
(a dropped term, a transposed operand, truncation, ties away from zero, an fp32
running sum) and checks that at least one pin fails for each.

The definition pinned is D[m,n] = RNE_fp16(sum_k A[m,k]·B[n,k]) with B stored
N×K ("GEMM I — the tiled baseline", "The problem we are solving"; the cast
happens once, at writeback, per Step 1's pseudocode).
"""
import bisect
from fractions import Fraction

import numpy as np
import pytest

import oracle

# --------------------------------------------------------------------------
# Independent fp16 reference: every finite non-negative fp16 value, exactly.
# --------------------------------------------------------------------------
_POS_BITS = np.arange(0x0000, 0x7C00, dtype=np.uint16)  # +0 ... 65504
_POS_VALS = [Fraction(float(v)) for v in _POS_BITS.view(np.float16).astype(np.float64)]


def exact_value(bits: int) -> Fraction:
    """Exact value of a finite fp16 bit pattern, via numpy's float16 (library)."""
    v = np.array([bits], dtype=np.uint16).view(np.float16).astype(np.float64)[0]
    assert np.isfinite(v)
    return Fraction(float(v))


def nearest_f16(x: Fraction) -> int:
    """Round an exact rational to fp16 by searching the table of all values.

    Nearest wins; an exact tie goes to the pattern with an even last bit; at or
    beyond 65520 (the midpoint past the largest finite value) the result is Inf.
    """
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    if a >= 65520:
        return sign | 0x7C00
    i = bisect.bisect_left(_POS_VALS, a)
    if i < len(_POS_VALS) and _POS_VALS[i] == a:
        return sign | int(_POS_BITS[i]) if a != 0 else 0
    lo, hi = i - 1, i
    if hi >= len(_POS_VALS):  # between 65504 and 65520
        return sign | int(_POS_BITS[lo])
    dlo, dhi = a - _POS_VALS[lo], _POS_VALS[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if int(_POS_BITS[lo]) % 2 == 0 else hi
    return sign | int(_POS_BITS[pick])


def exact_gemm(A_bits: np.ndarray, B_bits: np.ndarray):
    """Exact D = A·Bᵀ as Fractions (brute force, tiny inputs only)."""
    M, K = A_bits.shape
    N = B_bits.shape[0]
    a = [[exact_value(int(A_bits[m, k])) for k in range(K)] for m in range(M)]
    b = [[exact_value(int(B_bits[n, k])) for k in range(K)] for n in range(N)]
    return [[sum((a[m][k] * b[n][k] for k in range(K)), Fraction(0)) for n in range(N)] for m in range(M)]


def f16_bits(values) -> np.ndarray:
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def random_grid_f16(rng, shape, denom=256):
    """fp16 values j/denom with |j| <= denom: sums of a few products stay exact in fp64."""
    j = rng.integers(-denom, denom + 1, size=shape)
    return f16_bits(j / denom)


def random_wide_f16(rng, shape, lo_exp=-10, hi_exp=4):
    """fp16 values with random sign, exponent in [lo_exp, hi_exp] and random fraction."""
    e = rng.integers(lo_exp, hi_exp + 1, size=shape)
    f = rng.integers(0, 1024, size=shape)
    s = rng.integers(0, 2, size=shape)
    bits = (s << 15) | ((e + 15) << 10) | f
    return bits.astype(np.uint16)


# --------------------------------------------------------------------------
# Pins, written as predicates so that the planted-mistake test can reuse them.
# --------------------------------------------------------------------------

def pin_decode_exhaustive(mutant=0):
    allbits = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_to_f64(allbits, mutant=mutant)
    ref = allbits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    return bool(np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])
                and np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])))


def pin_encode_roundtrip(mutant=0):
    allbits = np.arange(65536, dtype=np.uint16)
    vals = allbits.view(np.float16).astype(np.float64)
    back = oracle.f64_to_f16(vals, mutant=mutant)
    finite = np.isfinite(vals) | np.isinf(vals)
    ok = np.array_equal(back[finite], allbits[finite])
    nan_back = back[~finite]
    ok &= bool(np.all(((nan_back & 0x7C00) == 0x7C00) & ((nan_back & 0x03FF) != 0)))
    return bool(ok)


def pin_encode_ties(mutant=0):
    """Every midpoint between adjacent finite fp16 values rounds to the even one."""
    lo = np.arange(0x0000, 0x7BFF, dtype=np.uint16)
    hi = lo + 1
    vlo = lo.view(np.float16).astype(np.float64)
    vhi = hi.view(np.float16).astype(np.float64)
    mid = (vlo + vhi) / 2  # exact: the midpoint needs 12 significant bits
    want = np.where(lo % 2 == 0, lo, hi).astype(np.uint16)
    got = oracle.f64_to_f16(mid, mutant=mutant)
    below = oracle.f64_to_f16(np.nextafter(mid, -np.inf), mutant=mutant)
    above = oracle.f64_to_f16(np.nextafter(mid, np.inf), mutant=mutant)
    neg = oracle.f64_to_f16(-mid, mutant=mutant)
    return bool(np.array_equal(got, want) and np.array_equal(below, lo) and np.array_equal(above, hi)
                and np.array_equal(neg, want | 0x8000))


def pin_encode_edges(mutant=0):
    cases = [
        (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00), (1e300, 0x7C00), (-65520.0, 0xFC00),
        (np.inf, 0x7C00), (-np.inf, 0xFC00), (0.0, 0x0000), (-0.0, 0x8000),
        (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (np.nextafter(2.0 ** -25, 1), 0x0001),
        (3 * 2.0 ** -25, 0x0002), (2.0 ** -14, 0x0400), (2.0 ** -14 - 2.0 ** -25, 0x0400),
        (1.0, 0x3C00), (1.0 + 2.0 ** -11, 0x3C00), (1.0 + 3 * 2.0 ** -11, 0x3C02), (2049.0, 0x6800),
        (2051.0, 0x6802), (1e-300, 0x0000),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float64)
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    return bool(np.array_equal(oracle.f64_to_f16(x, mutant=mutant), want))


def pin_encode_random_vs_numpy(mutant=0):
    """numpy's own double->half conversion (library routine) on many random doubles."""
    rng = np.random.default_rng(1234)
    x = rng.standard_normal(200_000) * np.exp2(rng.integers(-30, 17, size=200_000))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = oracle.f64_to_f16(x, mutant=mutant)
    sample = rng.choice(x.size, 300, replace=False)  # and a few against the exact table search
    ok_table = all(int(got[i]) == nearest_f16(Fraction(float(x[i]))) for i in sample)
    return bool(np.array_equal(got, ref) and ok_table)


def pin_identity_A(mutant=0):
    """A = I (M = K): D = Bᵀ exactly."""
    rng = np.random.default_rng(5)
    K, N = 16, 24
    A = f16_bits(np.eye(K))
    B = f16_bits(rng.uniform(-4, 4, size=(N, K)))
    D = oracle.gemm_f16_nt(A, B, mutant=mutant)
    return bool(np.array_equal(D, B.T))


def pin_identity_B(mutant=0):
    """B = I (N = K): D = A exactly."""
    rng = np.random.default_rng(6)
    M, K = 24, 16
    A = f16_bits(rng.uniform(-4, 4, size=(M, K)))
    B = f16_bits(np.eye(K))
    D = oracle.gemm_f16_nt(A, B, mutant=mutant)
    return bool(np.array_equal(D, A))


def pin_all_ones(mutant=0):
    """All-ones operands: D = K, rounded once (2049 -> 2048 and 2051 -> 2052 are ties)."""
    ok = True
    for K in (1, 7, 64, 2048, 2049, 2051, 4096):
        A = f16_bits(np.ones((3, K)))
        B = f16_bits(np.ones((5, K)))
        D = oracle.gemm_f16_nt(A, B, mutant=mutant)
        ok &= bool(np.all(D == nearest_f16(Fraction(K))))
    return ok


def pin_cancellation(mutant=0):
    """big + small - big = small: the running sum must hold more than fp32's 24 bits.

    Row [2048, 2^-7, -2048] against [1, 2^-6, 1] sums to exactly 2^-13 (an fp16
    normal); an fp32 accumulator drops the 2^-13 (half an ulp of 2048, tie to
    even) and returns 0.
    """
    A = f16_bits([[2048.0, 2.0 ** -7, -2048.0], [-1024.0, 2.0 ** -9, 1024.0]])
    B = f16_bits([[1.0, 2.0 ** -6, 1.0], [1.0, 2.0 ** -7, 1.0]])
    D = oracle.gemm_f16_nt(A, B, mutant=mutant)
    want = np.array([[nearest_f16(Fraction(2048) * 1 + Fraction(1, 2 ** 13) - 2048),
                      nearest_f16(Fraction(1, 2 ** 14))],
                     [nearest_f16(Fraction(1, 2 ** 15)), nearest_f16(Fraction(1, 2 ** 16))]], dtype=np.uint16)
    return bool(np.array_equal(D, want) and D[0, 0] == 0x0800)


def pin_rank1(mutant=0):
    """A[m,k] = a_m·[k=0], B[n,k] = b_n·[k=0]: D = RNE(a_m·b_n)."""
    rng = np.random.default_rng(7)
    M, N, K = 9, 11, 5
    a = random_wide_f16(rng, (M,), -8, 3)
    b = random_wide_f16(rng, (N,), -8, 3)
    A = np.zeros((M, K), dtype=np.uint16)
    B = np.zeros((N, K), dtype=np.uint16)
    A[:, 0], B[:, 0] = a, b
    D = oracle.gemm_f16_nt(A, B, mutant=mutant)
    want = np.array([[nearest_f16(exact_value(int(a[m])) * exact_value(int(b[n]))) for n in range(N)]
                     for m in range(M)], dtype=np.uint16)
    return bool(np.array_equal(D, want))


def pin_brute_force_exact(mutant=0):
    """Tiny grids of j/256 values: the fp64 sum is exact, so D must equal the exact sum rounded once."""
    rng = np.random.default_rng(8)
    for M, N, K in [(1, 1, 1), (2, 3, 5), (8, 8, 8), (7, 5, 3), (3, 8, 6), (5, 2, 8)]:
        A = random_grid_f16(rng, (M, K))
        B = random_grid_f16(rng, (N, K))
        D, acc = oracle.gemm_f16_nt(A, B, with_acc=True, mutant=mutant)
        ex = exact_gemm(A, B)
        want = np.array([[nearest_f16(v) for v in row] for row in ex], dtype=np.uint16)
        if not np.array_equal(D, want):
            return False
        if not all(Fraction(float(acc[m, n])) == ex[m][n] for m in range(M) for n in range(N)):
            return False
    return True


def pin_brute_force_wide(mutant=0):
    """Wide-exponent inputs: the fp64 sum is within a few fp64 ulps of exact; D equals exact rounding."""
    rng = np.random.default_rng(9)
    for M, N, K in [(4, 4, 8), (6, 3, 7), (8, 8, 4)]:
        A = random_wide_f16(rng, (M, K))
        B = random_wide_f16(rng, (N, K))
        D, acc = oracle.gemm_f16_nt(A, B, with_acc=True, mutant=mutant)
        ex = exact_gemm(A, B)
        for m in range(M):
            for n in range(N):
                mag = sum(abs(exact_value(int(A[m, k])) * exact_value(int(B[n, k]))) for k in range(K))
                if abs(Fraction(float(acc[m, n])) - ex[m][n]) > mag * K * Fraction(1, 2 ** 52):
                    return False
                if int(D[m, n]) != nearest_f16(ex[m][n]):
                    return False
    return True


def pin_invariants(mutant=0):
    """Swapping A and B transposes D bit for bit; negating A negates D."""
    rng = np.random.default_rng(10)
    A = f16_bits(rng.uniform(-1, 1, size=(13, 37)))
    B = f16_bits(rng.uniform(-1, 1, size=(19, 37)))
    D = oracle.gemm_f16_nt(A, B, mutant=mutant)
    Dt = oracle.gemm_f16_nt(B, A, mutant=mutant)
    Dn = oracle.gemm_f16_nt(A ^ np.uint16(0x8000), B, mutant=mutant)
    v, vn = D.view(np.float16).astype(np.float64), Dn.view(np.float16).astype(np.float64)
    return bool(np.array_equal(D, Dt.T) and np.array_equal(vn, -v))


PINS = [pin_decode_exhaustive, pin_encode_roundtrip, pin_encode_ties, pin_encode_edges,
        pin_encode_random_vs_numpy, pin_identity_A, pin_identity_B, pin_all_ones, pin_cancellation, pin_rank1,
        pin_brute_force_exact, pin_brute_force_wide, pin_invariants]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin(0)


# The mutants and the pins expected to catch each; test_planted_mistakes_are_caught
# only requires that some pin fails.
MUTANTS = {
    1: "last term of the contraction dropped",
    2: "B read as K×N (transposed operand)",
    3: "truncation instead of round-to-nearest-even",
    4: "ties rounded away from zero",
    5: "fp32 running sum",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_planted_mistakes_are_caught(mutant):
    failed = [p.__name__ for p in PINS if not p(mutant)]
    assert failed, f"no pin caught mutant {mutant} ({MUTANTS[mutant]})"


def test_points_match_full():
    rng = np.random.default_rng(11)
    A = f16_bits(rng.uniform(-1, 1, size=(33, 70)))
    B = f16_bits(rng.uniform(-1, 1, size=(21, 70)))
    D, acc = oracle.gemm_f16_nt(A, B, with_acc=True)
    rows = rng.integers(0, 33, size=200)
    cols = rng.integers(0, 21, size=200)
    p, pacc = oracle.gemm_f16_nt_points(A, B, rows, cols, with_acc=True, threads=3)
    assert np.array_equal(p, D[rows, cols])
    assert np.array_equal(pacc, acc[rows, cols])
    with pytest.raises(RuntimeError):
        oracle.gemm_f16_nt_points(A, B, [33], [0])


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(12)
    A = f16_bits(rng.uniform(-1, 1, size=(50, 64)))
    B = f16_bits(rng.uniform(-1, 1, size=(40, 64)))
    assert np.array_equal(oracle.gemm_f16_nt(A, B, threads=1), oracle.gemm_f16_nt(A, B, threads=7))


def test_degenerate_shapes():
    A = np.zeros((0, 8), dtype=np.uint16)
    B = np.zeros((4, 8), dtype=np.uint16)
    assert oracle.gemm_f16_nt(A, B).shape == (0, 4)
    # K = 0: the empty sum is +0
    D = oracle.gemm_f16_nt(np.zeros((3, 0), np.uint16), np.zeros((2, 0), np.uint16))
    assert D.shape == (3, 2) and np.all(D == 0)
