"""Randomised GPU parity: seeded random shapes, variants and entry points against the oracle.

Each case draws M (any), N and K (multiples of 8, the supported set), a kernel
variant (default, CTA pair, single CTA, two consumers; further series the
narrow 128 x 64 and the tiny 64 x 64 tiles, and narrow or tiny tiles with K
split across clusters of 2, 4 or 8 CTAs), a cap on the number of
persistent clusters (so that tail splits and multi-tile CTAs occur at small
sizes) and an entry point (no workspace, caller workspace, the library's fixed
scratch).  Every element must meet |gpu - oracle| <= 2^-9 |oracle| + 1e-3.

GEMM_FUZZ_CASES and GEMM_FUZZ_SEED (environment) change the number of cases of
the first series and the seed, and GEMM_FUZZ_SERIES_CASES the number of cases of
each of the narrow, tiny and K-split series, for longer sweeps; the defaults are
36, 2026 and 12.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as si

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _cases(n=36, seed=2026, per_series=12):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 1200))
        N = int(rng.integers(1, 150)) * 8
        K = int(rng.choice([int(rng.integers(1, 64)) * 8, int(rng.integers(64, 400)) * 8]))
        variant = [(0, 0), (2, 1), (1, 1), (2, 2)][int(rng.integers(0, 4))]
        clusters = int(rng.choice([0, 0, 1, 2, 3, 5, 7, 16]))
        entry = ["nt", "ws", "static"][int(rng.integers(0, 3))]
        out.append((i, M, N, K, variant, clusters, entry))
    # make sure split-K (few tiles, long K) shows up with each workspace entry point
    out.append((n, 256, 264, 2600, (2, 1), 0, "ws"))  # the default would take narrow tiles here
    out.append((n + 1, 500, 512, 2048, (1, 1), 0, "static"))
    # narrow, tiny and thin tiles, forced, with the K-loop both inside and beyond
    # the 8- and 12-stage rings
    for series, variant in ((1, (1, 1, 64, 128)), (2, (1, 1, 64, 64)), (3, None), (4, (1, 1, 16, 64))):
        rng = np.random.default_rng(seed + series)
        first = n + 2 + per_series * (series - 1)
        for i in range(first, first + per_series):
            M = int(rng.integers(1, 700))
            N = int(rng.integers(1, 100)) * 8
            K = int(rng.integers(1, 130)) * 8
            clusters = int(rng.choice([0, 0, 1, 3, 7]))
            entry = ["nt", "ws", "static"][int(rng.integers(0, 3))]
            v = variant if variant is not None else (1, 1, 64, int(rng.choice([64, 128])), int(rng.choice([2, 4, 8])))
            out.append((i, M, N, K, v, clusters, entry))
    return out


@pytest.mark.parametrize("i,M,N,K,variant,clusters,entry",
                         _cases(int(os.environ.get("GEMM_FUZZ_CASES", "36")), int(os.environ.get("GEMM_FUZZ_SEED", "2026")),
                                int(os.environ.get("GEMM_FUZZ_SERIES_CASES", "12"))),
                         ids=lambda v: str(v) if isinstance(v, int) else None)
def test_random_case(gpu_lib, i, M, N, K, variant, clusters, entry):
    lib = gpu_lib.load()
    A, B = si.custom(M, N, K, seed=1000 + i).operands()
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    o = gpu_lib.Options(cta_group=variant[0], consumers=variant[1], max_clusters=clusters,
                        block_n=variant[2] if len(variant) > 2 else 0, block_m=variant[3] if len(variant) > 3 else 0,
                        cluster_k=variant[4] if len(variant) > 4 else 0)
    stream = torch.cuda.current_stream().cuda_stream
    if entry == "nt":
        rc = gpu_lib.gemm_f16_nt_ptr(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), M, N, K, stream, o)
    elif entry == "ws":
        need = gpu_lib.workspace_size(M, N, K, o)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        rc = gpu_lib.gemm_f16_nt_ptr(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), M, N, K, stream, o,
                                     ws.data_ptr(), need)
    else:
        rc = lib.gemm_f16_nt_static_ws(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), M, N, K, stream,
                                       ctypes.byref(o))
        if rc == -9:
            pytest.skip("split-K scratch larger than the fixed array")
    assert rc == 0, gpu_lib.status_string(rc)
    status, info = gpu_lib.last_device_status()
    assert status == 0, f"{gpu_lib.status_string(status)} info={info:#x}"
    got = D.cpu().numpy().astype(np.float64)
    ref = oracle.gemm_f16_nt(A, B).view(np.float16).astype(np.float64)
    bad = ~(np.abs(got - ref) <= 2.0 ** -9 * np.abs(ref) + 1e-3)
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} elements off; first at {np.argwhere(bad)[0]}"
