"""gemm_f16_nt_static_ws: the GEMM entry point that allocates nothing, called through the C ABI.

Some callers cannot allocate device memory while they run: code that fixes its
memory budget once and forbids later allocation, a plug-in living inside an
application that owns the GPU's memory, or a loop where an allocation (which
may block and synchronise the device) is not allowed.  This entry point gives
them split-K using a fixed 16 MiB scratch array inside the library instead of
a workspace they would have to allocate.

The checks:
- on two shapes whose launch splits K over CTA pairs (so the fixed array is
  really used; gemm_f16_nt_describe says so), the results match the CPU oracle
  within the tolerance of the other GPU tests, and match the entry point that
  takes a caller-owned workspace (gemm_f16_nt_ws), on two calls in a row (the
  second finds the first call's leftovers in the shared array);
- further calls leave the device's free memory (cudaMemGetInfo) unchanged;
- a problem that needs no scratch runs as usual;
- a problem whose scratch would not fit is refused before anything runs.
"""
import ctypes

import numpy as np
import pytest

import oracle
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
    return gpu_lib.Options(cta_group=2)


def _static_call(lib, A, B, D, M, N, K, opts=None):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.gemm_f16_nt_static_ws(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                     ctypes.c_void_p(D.data_ptr()), M, N, K, ctypes.c_void_p(stream),
                                     ctypes.byref(opts) if opts is not None else None)


def _workspace_call(lib, A, B, D, M, N, K, opts=None):
    o = ctypes.byref(opts) if opts is not None else None
    need = lib.gemm_f16_nt_workspace_size(M, N, K, o)
    assert need >= 0
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gemm_f16_nt_ws(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                            ctypes.c_void_p(D.data_ptr()), M, N, K, ctypes.c_void_p(ws.data_ptr()), need,
                            ctypes.c_void_p(stream), o)
    torch.cuda.synchronize()
    return rc


def _assert_close(got, ref, what):
    g = np.asarray(got, dtype=np.float16).astype(np.float64)
    r = np.asarray(ref).view(np.float16).astype(np.float64) if np.asarray(ref).dtype == np.uint16 else \
        np.asarray(ref, dtype=np.float16).astype(np.float64)
    ok = np.abs(g - r) <= RTOL * np.abs(r) + ATOL
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} elements outside |d| <= 2^-9 |ref| + 1e-3"


SHAPES = [(768, 640, 4096), (512, 1024, 4096)]  # both split K over CTA pairs: 15 and 16 MiB of scratch


def test_static_scratch_matches_the_oracle_and_the_workspace_entry_point(gpu_lib):
    lib = gpu_lib.load()
    probs = []
    for i, (M, N, K) in enumerate(SHAPES):
        cfg = gpu_lib.describe(M, N, K, _pairs(gpu_lib), with_workspace=True)
        assert cfg["split_k"] > 1, f"{M}x{N}x{K} is meant to split K, so that the fixed array is used"
        need = lib.gemm_f16_nt_workspace_size(M, N, K, ctypes.byref(_pairs(gpu_lib)))
        assert 0 < need <= STATIC_BYTES and need == cfg["workspace_bytes"]
        A, B = si.custom(M, N, K, seed=90 + i).operands()
        probs.append((M, N, K, A, B, _dev(A), _dev(B)))
    # two calls in a row through the fixed scratch, the second on top of the first's leftovers
    outs = []
    for M, N, K, _, _, dA, dB in probs:
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _static_call(lib, dA, dB, D, M, N, K, _pairs(gpu_lib)) == 0
        outs.append(D)
    torch.cuda.synchronize()
    assert gpu_lib.last_device_status()[0] == 0
    for (M, N, K, A, B, dA, dB), D in zip(probs, outs):
        got = D.cpu().numpy()
        _assert_close(got, oracle.gemm_f16_nt(A, B), f"static scratch {M}x{N}x{K} against the oracle")
        ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
        assert _workspace_call(lib, dA, dB, ref, M, N, K, _pairs(gpu_lib)) == 0
        _assert_close(got, ref.cpu().numpy(), f"static scratch {M}x{N}x{K} against gemm_f16_nt_ws")


def test_static_scratch_calls_allocate_no_device_memory(gpu_lib):
    lib = gpu_lib.load()
    probs = []
    for i, (M, N, K) in enumerate(SHAPES):
        A, B = si.custom(M, N, K, seed=80 + i).operands()
        D = torch.empty((M, N), dtype=torch.float16, device="cuda")
        probs.append((M, N, K, _dev(A), _dev(B), D))
    for M, N, K, dA, dB, D in probs:  # first calls: per-device set-up and the kernels' first loads
        assert _static_call(lib, dA, dB, D, M, N, K, _pairs(gpu_lib)) == 0
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(4):
        for M, N, K, dA, dB, D in probs:
            assert _static_call(lib, dA, dB, D, M, N, K, _pairs(gpu_lib)) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert gpu_lib.last_device_status()[0] == 0
    assert free_after == free_before, f"free device memory changed by {free_before - free_after} bytes"


def test_static_scratch_without_split_k(gpu_lib):
    lib = gpu_lib.load()
    M, N, K = 1536, 1536, 512  # enough tiles: no split-K, no scratch used
    assert lib.gemm_f16_nt_workspace_size(M, N, K, None) == 0
    A, B = si.custom(M, N, K, seed=95).operands()
    dA, dB = _dev(A), _dev(B)
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    assert _static_call(lib, dA, dB, D, M, N, K) == 0
    torch.cuda.synchronize()
    assert gpu_lib.last_device_status()[0] == 0
    _assert_close(D.cpu().numpy(), oracle.gemm_f16_nt(A, B), "no split-K")


def test_static_scratch_refuses_what_does_not_fit(gpu_lib):
    lib = gpu_lib.load()
    # few-tile, long-K shapes over CTA pairs; on GB300 (76 co-resident pairs) the first needs
    # 8 slices x 768 x 768 x 4 B = 18 MiB of scratch.  Devices with other pair counts cut K
    # into other slice counts, so look for a shape that needs more than the array holds.
    candidates = [(768, 768, 4096), (768, 1024, 4096), (1280, 768, 4096), (1024, 1024, 8192), (1536, 1024, 8192),
                  (2048, 1024, 8192), (2048, 2048, 16384)]
    big = None
    for M, N, K in candidates:
        need = lib.gemm_f16_nt_workspace_size(M, N, K, ctypes.byref(_pairs(gpu_lib)))
        if need > STATIC_BYTES:
            big = (M, N, K)
            break
    assert big is not None, "no candidate shape needs more scratch than the fixed array holds"
    M, N, K = big
    A, B = si.custom(M, N, K, seed=96).operands()
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    assert _static_call(lib, _dev(A), _dev(B), D, M, N, K, _pairs(gpu_lib)) == SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.isnan(D).all()  # nothing ran
    assert "16 MiB" in gpu_lib.status_string(SCRATCH_LIMIT)
