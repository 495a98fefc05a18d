"""The checked build: the same library compiled with its device range checks.

Instead of an external memory checker, the kernel carries its own range
checks, compiled in only for the checked library (-DGEMM_F16_DEVICE_CHECKS=1):
every work item the scheduler hands out, every ring stage, the TMEM columns of
each accumulator, the epilogue's chunk count and staging buffer, and the rows a
CTA adds up when K is split across a cluster.  A failed
check would end the kernel with GEMM_ERR_DEVICE_BOUNDS in the status word
(never a trap).  Every kernel variant runs here through that build, over tile
grids, ragged edges, split tails, split-K and few persistent clusters: no
check may fail, and D must equal, bit for bit, what the production build
computes (the checks do not touch the arithmetic).
"""
import ctypes

import numpy as np
import pytest

import oracle
import seeded_inputs as si

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

CASES = [
    # (M, N, K, cta_group, consumers, block_n, max_clusters, workspace[, block_m[, cluster_k]])
    (128, 128, 64, 0, 0, 0, 0, False),       # default: thin 64 x 16 tiles
    (256, 256, 512, 0, 0, 0, 0, False),      # default: thin tiles, a K-loop of 8 tiles
    (256, 256, 512, 0, 0, 64, 0, False, 64, 4),  # tiny tiles, K split across clusters of 4
    (700, 600, 1000, 1, 1, 16, 9, False, 64),  # thin tiles, many per CTA, K beyond the ring, ragged
    (200, 136, 520, 1, 1, 64, 0, False, 64, 8),   # K split over 8 CTAs, ragged M, N and K
    (520, 264, 1000, 1, 1, 64, 0, False, 64, 2),  # K split over 2 CTAs, K beyond the ring
    (300, 200, 1000, 1, 1, 64, 0, False, 128, 4),  # narrow tiles, K split over 4 CTAs, ragged
    (700, 600, 1000, 1, 1, 64, 5, False, 64),  # tiny tiles, many per CTA, K beyond the ring
    (1000, 520, 1000, 2, 1, 256, 3, False),  # pairs, many tiles per cluster, ragged
    (1000, 520, 1000, 1, 1, 256, 5, False),  # single CTAs
    (1000, 520, 1000, 2, 2, 256, 2, False),  # two consumers
    (700, 600, 2000, 1, 1, 64, 7, False),    # narrow tiles, K beyond the ring
    (2560, 1280, 512, 2, 1, 256, 7, False),  # tail split along N (50 tiles on 7 pairs)
    (256, 264, 2600, 2, 1, 256, 0, True),    # split-K through a workspace
    (4096, 4096, 4096, 0, 0, 0, 0, False),   # the headline shape
]


def _call(lib, dA, dB, M, N, K, o, ws):
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if ws is not None:
        rc = lib.gemm_f16_nt_ws(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), M, N, K, ws.data_ptr(), ws.numel(),
                                stream, ctypes.byref(o))
    else:
        rc = lib.gemm_f16_nt_ex(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), M, N, K, stream, ctypes.byref(o))
    assert rc == 0
    info = ctypes.c_uint64(0)
    status = lib.gemm_f16_last_device_status(stream, ctypes.byref(info))
    return D, status, info.value


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(v) for v in c[:3]) + f"-cg{c[3]}-nc{c[4]}-bn{c[5]}"
                         + (f"-bm{c[8]}" if len(c) > 8 else "") + (f"-ck{c[9]}" if len(c) > 9 else ""))
def test_checked_build_runs_clean_and_matches(gpu_lib, case):
    M, N, K, cg, nc, bn, clusters, use_ws = case[:8]
    checked, prod = gpu_lib.load_checked(), gpu_lib.load()
    o = gpu_lib.Options(cta_group=cg, consumers=nc, block_n=bn, max_clusters=clusters,
                        block_m=case[8] if len(case) > 8 else 0, cluster_k=case[9] if len(case) > 9 else 0)
    A, B = si.custom(M, N, K, seed=M + 2 * N + 3 * K).operands()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    ws = None
    if use_ws:
        need = gpu_lib.workspace_size(M, N, K, o)
        assert need > 0
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    Dc, status, info = _call(checked, dA, dB, M, N, K, o, ws)
    assert status == 0, f"{gpu_lib.status_string(status)} info={info:#x}"
    Dp, status_p, _ = _call(prod, dA, dB, M, N, K, o, ws)
    assert status_p == 0
    assert torch.equal(Dc.view(torch.int16), Dp.view(torch.int16)), "checked and production builds differ"
    if M * N * K <= 1 << 30:
        got = Dc.cpu().numpy().astype(np.float64)
        ref = oracle.gemm_f16_nt(A, B).view(np.float16).astype(np.float64)
        assert np.all(np.abs(got - ref) <= 2.0 ** -9 * np.abs(ref) + 1e-3)
