"""gemm_f16_nt_static_ws: the GEMM entry point that allocates nothing, called through the C ABI.

Some callers cannot allocate device memory while they run: code that fixes its
memory budget once and forbids later allocation, a plug-in living inside an
application that owns the GPU's memory, or a loop where an allocation (which
may block and synchronise the device) is not allowed.  This entry point gives
them split-K using a fixed 16 MiB scratch array inside the library instead of
a workspace they would have to allocate.

The checks: its results match those of the entry point that takes a
caller-owned workspace (gemm_f16_nt_ws), within the tolerance the other GPU
tests use, on two calls in a row (the second finds the first call's leftovers
in the shared array); a problem that needs no scratch runs as usual; and a
problem whose scratch would not fit is refused before anything runs.
"""
import ctypes

import numpy as np
import pytest

import seeded_inputs as si

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

RTOL = 2.0 ** -9
ATOL = 1e-3
SCRATCH_LIMIT = -9
STATIC_BYTES = 16 << 20


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _pairs(gpu_lib):
    # CTA pairs: their split-K uses scratch (by default these long-K shapes would instead split
    # K across thread-block clusters, which needs none)
    return ctypes.byref(gpu_lib.Options(cta_group=2))


def _static_call(lib, A, B, D, M, N, K, opts=None):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.gemm_f16_nt_static_ws(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                     ctypes.c_void_p(D.data_ptr()), M, N, K, ctypes.c_void_p(stream), opts)


def _workspace_call(lib, A, B, D, M, N, K, opts=None):
    need = lib.gemm_f16_nt_workspace_size(M, N, K, opts)
    assert need >= 0
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gemm_f16_nt_ws(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                            ctypes.c_void_p(D.data_ptr()), M, N, K, ctypes.c_void_p(ws.data_ptr()), need,
                            ctypes.c_void_p(stream), opts)
    torch.cuda.synchronize()
    return rc


def _close(got, ref):
    g = got.cpu().numpy().astype(np.float64)
    r = ref.cpu().numpy().astype(np.float64)
    return bool(np.all(np.abs(g - r) <= RTOL * np.abs(r) + ATOL))


def test_static_scratch_matches_the_workspace_entry_point(gpu_lib):
    lib = gpu_lib.load()
    shapes = [(768, 640, 4096), (512, 1024, 4096)]  # both split K (15 MiB and 16 MiB of scratch)
    probs = []
    for i, (M, N, K) in enumerate(shapes):
        assert 0 < lib.gemm_f16_nt_workspace_size(M, N, K, _pairs(gpu_lib)) <= STATIC_BYTES
        A, B = si.custom(M, N, K, seed=90 + i).operands()
        probs.append((M, N, K, _dev(A), _dev(B)))
    # two calls in a row through the fixed scratch, the second on top of the first's leftovers
    outs = []
    for M, N, K, A, B in probs:
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _static_call(lib, A, B, D, M, N, K, _pairs(gpu_lib)) == 0
        outs.append(D)
    torch.cuda.synchronize()
    assert gpu_lib.last_device_status()[0] == 0
    for (M, N, K, A, B), D in zip(probs, outs):
        ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
        assert _workspace_call(lib, A, B, ref, M, N, K, _pairs(gpu_lib)) == 0
        assert _close(D, ref), f"{M}x{N}x{K}"


def test_static_scratch_without_split_k(gpu_lib):
    lib = gpu_lib.load()
    M, N, K = 1536, 1536, 512  # enough tiles: no split-K, no scratch used
    assert lib.gemm_f16_nt_workspace_size(M, N, K, None) == 0
    A, B = si.custom(M, N, K, seed=95).operands()
    dA, dB = _dev(A), _dev(B)
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    assert _static_call(lib, dA, dB, D, M, N, K) == 0
    ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert _workspace_call(lib, dA, dB, ref, M, N, K) == 0
    assert _close(D, ref)


def test_static_scratch_refuses_what_does_not_fit(gpu_lib):
    lib = gpu_lib.load()
    M, N, K = 768, 768, 4096  # 9 pair tiles, 8 K slices: 8 x 768 x 768 x 4 B = 18 MiB of scratch
    need = lib.gemm_f16_nt_workspace_size(M, N, K, _pairs(gpu_lib))
    if need <= STATIC_BYTES:
        pytest.skip(f"on this device the shape needs only {need} bytes")
    A, B = si.custom(M, N, K, seed=96).operands()
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    assert _static_call(lib, _dev(A), _dev(B), D, M, N, K, _pairs(gpu_lib)) == SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.isnan(D).all()  # nothing ran
    assert "16 MiB" in gpu_lib.status_string(SCRATCH_LIMIT)
