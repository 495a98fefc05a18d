"""GPU parity: the sm_103a kernel, called through the C ABI, against the CPU oracle.

Bar (per element, floating point): |gpu − oracle| ≤ 2⁻⁹·|oracle| + 1e-3, with
the oracle the fp64 sum rounded once to fp16.  Cases with one product per
output (identity operands) must match bit for bit.

Every shape is compared in full, the three large workloads (4096³, 8192³,
8192×28672×4096) included, in the launch configuration the benchmark times and
with two MMA consumers.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as si

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

RTOL = 2.0 ** -9
ATOL = 1e-3
SENTINEL = 0x7E00  # an fp16 NaN no finite result can equal


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run(g, A, B, options=None):
    D = g.gemm_f16_nt(to_dev(A), to_dev(B), options=options)
    status, info = g.last_device_status()
    assert status == 0, f"device status {g.status_string(status)} info={info:#x}"
    return D.cpu().numpy()


def assert_close(gpu_f16, ref_bits, what=""):
    got = np.asarray(gpu_f16, dtype=np.float16).astype(np.float64)
    ref = np.asarray(ref_bits).view(np.float16).astype(np.float64)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    ok = err <= RTOL * np.abs(ref) + ATOL
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} outside tolerance; first at {i}: "
                             f"gpu={got[i]!r} oracle={ref[i]!r}")


# (cta_group, consumers, block_n[, block_m[, cluster_k]]): the CTA pair with
# one MMA consumer (the default), a single CTA, the pair with two consumers
# sharing each B stage, the narrow 128 x 64 single-CTA tiles of small problems
# and the tiny 64 x 64 tiles (MMAs of M = 64) of the smallest, each without a K
# split and with K split across clusters of 2, 4 and 8 CTAs (fewer where K has
# fewer 64-wide tiles), and the thin 64 x 16 tiles (MMAs of M = 64, N = 16).
VARIANTS = [(2, 1, 256), (1, 1, 256), (2, 2, 256), (1, 1, 64, 128, 1), (1, 1, 64, 128, 2), (1, 1, 64, 128, 4),
            (1, 1, 64, 128, 8), (1, 1, 64, 64, 1), (1, 1, 64, 64, 2), (1, 1, 64, 64, 4), (1, 1, 64, 64, 8),
            (1, 1, 16, 64, 1)]
VIDS = ["pair", "single", "pair-2consumers", "narrow", "narrow-k2", "narrow-k4", "narrow-k8", "tiny", "tiny-k2",
        "tiny-k4", "tiny-k8", "thin"]


def opts(g, variant=(0, 0), max_clusters=0):
    return g.Options(cta_group=variant[0], max_clusters=max_clusters, consumers=variant[1],
                     block_n=variant[2] if len(variant) > 2 else 0, block_m=variant[3] if len(variant) > 3 else 0,
                     cluster_k=variant[4] if len(variant) > 4 else 0)


# ----------------------------------------------------------- full compares --

@pytest.mark.parametrize("v", VARIANTS + [(0, 0)], ids=VIDS + ["default"])
@pytest.mark.parametrize("name", ["single_tile_128x128x64", "ktile_grid_256x256x512"])
def test_small_workloads_full(gpu_lib, name, v):
    w = si.WORKLOADS[name]
    A, B = w.operands()
    assert_close(run(gpu_lib, A, B, opts(gpu_lib, v)), oracle.gemm_f16_nt(A, B), f"{name} {v}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 4096), (128, 128, 4096), (128, 1024, 1024), (200, 136, 3000)])
def test_default_cluster_k_split_full(gpu_lib, M, N, K):
    # small outputs with a long K take tiny tiles with K split across a cluster by default
    ks = gpu_lib.describe(M, N, K)["cluster_k"]
    assert ks > 1, "this shape is meant to split K across a cluster"
    A, B = si.custom(M, N, K, seed=M + N + K + 5).operands()
    assert_close(run(gpu_lib, A, B), oracle.gemm_f16_nt(A, B), f"{M}x{N}x{K} cluster_k={ks}")


@pytest.mark.parametrize("v", VARIANTS, ids=VIDS)
def test_identity_operands_are_exact(gpu_lib, v):
    # One product per output element: the result is exact, so bit equality.
    # A = I (M = K = 384, 1.5 cluster tiles) gives D = Bᵀ; B = I gives D = A.
    rng = np.random.default_rng(21)
    K = 384
    B = rng.uniform(-2, 2, size=(520, K)).astype(np.float16)
    D = run(gpu_lib, np.eye(K, dtype=np.float16), B, opts(gpu_lib, v))
    assert np.array_equal(D.view(np.uint16), np.ascontiguousarray(B.T).view(np.uint16))
    A = rng.uniform(-2, 2, size=(200, K)).astype(np.float16)
    D = run(gpu_lib, A, np.eye(K, dtype=np.float16), opts(gpu_lib, v))
    assert np.array_equal(D.view(np.uint16), A.view(np.uint16))


def _range_edge_operands(seed):
    """Row and column groups whose products put D in every fp16 range.

    A rows 0-63: +256·u, rows 64-127: −256·u (u in [0.5, 1)), rows 128-191:
    ±2⁻¹²·u, rows 192-255: ±u.  B columns 0-95: +256·v, columns 96-191:
    ±2⁻¹²·v.  With K = 320 the big rows times the big columns sum to at least
    5·10⁶ (±Inf in fp16), the tiny rows times the tiny columns to about 2⁻²¹
    (fp16 subnormals, below 2⁻¹⁴), and every other block stays finite.
    """
    rng = np.random.default_rng(seed)
    K = 320
    u = rng.uniform(0.5, 1.0, size=(256, K))
    sign = np.where(rng.random((256, K)) < 0.5, -1.0, 1.0)
    A = np.empty((256, K))
    A[0:64] = 256.0 * u[0:64]
    A[64:128] = -256.0 * u[64:128]
    A[128:192] = 2.0 ** -12 * u[128:192] * sign[128:192]
    A[192:256] = u[192:256] * sign[192:256]
    v = rng.uniform(0.5, 1.0, size=(192, K))
    vsign = np.where(rng.random((192, K)) < 0.5, -1.0, 1.0)
    B = np.empty((192, K))
    B[0:96] = 256.0 * v[0:96]
    B[96:192] = 2.0 ** -12 * v[96:192] * vsign[96:192]
    return A.astype(np.float16), B.astype(np.float16)


@pytest.mark.parametrize("v", VARIANTS + [(0, 0)], ids=VIDS + ["default"])
def test_range_edges_overflow_and_subnormals(gpu_lib, v):
    A, B = _range_edge_operands(5)
    got = run(gpu_lib, A, B, opts(gpu_lib, v))
    ref_bits = oracle.gemm_f16_nt(A, B)
    ref = ref_bits.view(np.float16).astype(np.float64)
    g64 = got.astype(np.float64)
    inf = np.isinf(ref)
    assert inf[0:128, 0:96].all() and not inf[128:].any(), "the operands do not reach the intended ranges"
    # overflow: the same infinity, bit for bit
    assert np.array_equal(got.view(np.uint16)[inf], ref_bits[inf]), f"{v}: infinities differ"
    # subnormal results of the tiny block (all products tiny, so fp32 accumulation error is far
    # below a subnormal step): within one step (2^-24), so a flush to zero would fail.  Elsewhere
    # a subnormal can arise from cancelling large products and only the usual bound applies.
    sub = np.zeros_like(inf)
    sub[128:192, 96:192] = (np.abs(ref[128:192, 96:192]) < 2.0 ** -14) & (ref[128:192, 96:192] != 0)
    assert sub[128:192, 96:192].mean() > 0.9, "the tiny block does not land in the subnormal range"
    assert np.all(np.abs(g64[sub] - ref[sub]) <= 2.0 ** -24), f"{v}: subnormal results off by more than one step"
    # everything finite within the usual bound
    fin = ~inf
    assert np.all(np.isfinite(g64[fin])), f"{v}: a finite result came out infinite"
    err = np.abs(g64[fin] - ref[fin])
    assert np.all(err <= RTOL * np.abs(ref[fin]) + ATOL), f"{v}: finite results outside tolerance"


RAGGED = [(1, 8, 8), (200, 136, 72), (129, 264, 520), (383, 1032, 1000), (1000, 8, 64), (640, 776, 8)]


@pytest.mark.parametrize("v", VARIANTS, ids=VIDS)
@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_shapes_full(gpu_lib, M, N, K, v):
    w = si.custom(M, N, K, seed=M * 7 + N * 3 + K)
    A, B = w.operands()
    assert_close(run(gpu_lib, A, B, opts(gpu_lib, v)), oracle.gemm_f16_nt(A, B), f"{M}x{N}x{K} {v}")


@pytest.mark.parametrize("v,clusters", [((2, 1), 1), ((2, 1), 3), ((1, 1), 1), ((1, 1), 5), ((2, 2), 1), ((2, 2), 3),
                                        ((1, 1, 64), 1), ((1, 1, 64), 6), ((1, 1, 64, 64), 1),
                                        ((1, 1, 64, 64), 7), ((1, 1, 16, 64), 1), ((1, 1, 16, 64), 9)])
def test_few_persistent_clusters_run_many_tiles(gpu_lib, v, clusters):
    # 1024 x 1024 x 320: 16 (pair), 32 (single CTA), 8 (two consumers), 128
    # (narrow), 256 (tiny) or 1024 (thin) tiles, so each persistent CTA runs
    # several tiles and both rings wrap many times across tiles.
    w = si.custom(1024, 1024, 320, seed=77)
    A, B = w.operands()
    assert_close(run(gpu_lib, A, B, opts(gpu_lib, v, clusters)), oracle.gemm_f16_nt(A, B),
                 f"{v} clusters={clusters}")


@pytest.mark.parametrize("M,N,K,v,clusters", [
    (1024, 1024, 320, (2, 1), 5),   # 16 tiles on 5 pairs: 15 whole + 1 split into halves
    (1024, 1024, 320, (1, 1), 30),  # 32 tiles on 30 CTAs: 2 split
    (640, 776, 200, (2, 1), 5),     # ragged N: a split half lies wholly past the last column
    (256, 4096, 512, (2, 1), 76),   # 16 tiles on 76 pairs: every tile split
    (1024, 1024, 320, (2, 1), 10),  # 16 % 10 = 6 > 10 / 2: no split
    (1024, 1024, 320, (2, 2), 3),   # two consumers: 8 tiles on 3 pairs, 2 split
    (640, 776, 200, (2, 2), 7),     # two consumers, ragged M and N, split halves past N
])
def test_split_last_wave(gpu_lib, M, N, K, v, clusters):
    w = si.custom(M, N, K, seed=M + N + K + v[0])
    A, B = w.operands()
    assert_close(run(gpu_lib, A, B, opts(gpu_lib, v, clusters)), oracle.gemm_f16_nt(A, B),
                 f"split {M}x{N}x{K} {v} clusters={clusters}")


@pytest.mark.parametrize("M,N,K,cg", [
    (256, 256, 4096, 2),     # one tile, 8 K slices
    (1024, 1024, 4096, 2),   # 16 tiles, 4 slices
    (256, 4096, 2048, 2),    # a skinny M: 16 tiles, 4 slices
    (300, 520, 3000, 2),     # ragged M, N and K: 6 tiles, 5 uneven slices
    (256, 256, 4096, 1),     # single-CTA tiles
])
def test_split_k_full(gpu_lib, M, N, K, cg):
    w = si.custom(M, N, K, seed=M + N + K)
    A, B = w.operands()
    o = gpu_lib.Options(cta_group=cg)
    need = gpu_lib.workspace_size(M, N, K, o)
    assert need > 0 and need % (4 * M * N) == 0, "this shape is meant to split K"
    dA, dB = to_dev(A), to_dev(B)
    # the workspace needs no initialisation: fill it with NaN
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device="cuda")
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    rc = gpu_lib.gemm_f16_nt_ptr(dA.data_ptr(), dB.data_ptr(), D.data_ptr(), M, N, K,
                                 torch.cuda.current_stream().cuda_stream, o, ws.data_ptr(), need)
    assert rc == 0
    assert gpu_lib.last_device_status()[0] == 0
    ref = oracle.gemm_f16_nt(A, B)
    assert_close(D.cpu().numpy(), ref, f"split-K {M}x{N}x{K} cg={cg}")
    # a workspace one byte too small: no split-K, same answer
    D2 = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    rc = gpu_lib.gemm_f16_nt_ptr(dA.data_ptr(), dB.data_ptr(), D2.data_ptr(), M, N, K,
                                 torch.cuda.current_stream().cuda_stream, o, ws.data_ptr(), need - 1)
    assert rc == 0 and gpu_lib.last_device_status()[0] == 0
    assert_close(D2.cpu().numpy(), ref, f"no split-K {M}x{N}x{K} cg={cg}")
    # the Python call supplies a workspace by itself
    assert_close(gpu_lib.gemm_f16_nt(dA, dB, options=o).cpu().numpy(), ref, "binding")


def test_binding_workspace_on_a_side_stream(gpu_lib):
    # The binding's cached split-K workspace belongs to the stream the call runs on; a larger
    # problem on the same stream replaces it while the first GEMM may still be queued.
    # (CTA pairs forced: by default these shapes split K across clusters, without a workspace)
    side = torch.cuda.Stream()
    pairs = gpu_lib.Options(cta_group=2)
    shapes = [(768, 640, 4096), (768, 768, 4096)]  # 15 MiB, then 18 MiB of partials
    outs = []
    for i, (M, N, K) in enumerate(shapes):
        assert gpu_lib.workspace_size(M, N, K, pairs) > 0
        A, B = si.custom(M, N, K, seed=700 + i).operands()
        dA, dB = to_dev(A), to_dev(B)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            D = gpu_lib.gemm_f16_nt(dA, dB, stream=side, options=pairs)
        outs.append((A, B, D))
    side.synchronize()
    assert gpu_lib.last_device_status(side.cuda_stream)[0] == 0
    for A, B, D in outs:
        assert_close(D.cpu().numpy(), oracle.gemm_f16_nt(A, B), f"side stream {A.shape[0]}x{B.shape[0]}")


def test_guard_bands_and_full_overwrite(gpu_lib):
    # D sits inside a larger buffer filled with a NaN sentinel: every element of
    # D must be written, and nothing before or after it.
    M, N, K = 300, 520, 200
    w = si.custom(M, N, K, seed=5)
    A, B = w.operands()
    guard = 32768
    buf = torch.full((guard + M * N + guard,), SENTINEL, dtype=torch.int16, device="cuda").view(torch.float16)
    D = buf[guard:guard + M * N].view(M, N)
    gpu_lib.gemm_f16_nt(to_dev(A), to_dev(B), D)
    status, _ = gpu_lib.last_device_status()
    assert status == 0
    host = buf.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(host[:guard] == SENTINEL) and np.all(host[guard + M * N:] == SENTINEL)
    assert not np.any(host[guard:guard + M * N] == SENTINEL)
    assert_close(host[guard:guard + M * N].view(np.float16).reshape(M, N), oracle.gemm_f16_nt(A, B), "guarded")


def test_degenerate_shapes(gpu_lib):
    # K = 0: every output is the empty sum, +0.
    D = torch.full((130, 264), 7.0, dtype=torch.float16, device="cuda")
    A = torch.empty((130, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((264, 0), dtype=torch.float16, device="cuda")
    gpu_lib.gemm_f16_nt(A, B, D)
    assert gpu_lib.last_device_status()[0] == 0
    assert torch.count_nonzero(D).item() == 0
    # M = 0 or N = 0: nothing to compute, nothing launched.
    E = gpu_lib.gemm_f16_nt(torch.empty((0, 64), dtype=torch.float16, device="cuda"),
                            torch.ones((8, 64), dtype=torch.float16, device="cuda"))
    assert tuple(E.shape) == (0, 8)


def test_argument_errors_on_device(gpu_lib):
    A = torch.ones((128, 64), dtype=torch.float16, device="cuda")
    B = torch.ones((128, 64), dtype=torch.float16, device="cuda")
    D = torch.zeros((128 * 128 + 8,), dtype=torch.float16, device="cuda")
    rc = gpu_lib.gemm_f16_nt_ptr(A.data_ptr(), B.data_ptr(), D.data_ptr() + 2, 128, 128, 64,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == -3
    rc = gpu_lib.gemm_f16_nt_ptr(A.data_ptr(), B.data_ptr(), D.data_ptr(), 128, 12, 64,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == -2
    assert torch.count_nonzero(D).item() == 0


@pytest.mark.parametrize("overlap", [1, -1])
def test_back_to_back_dependent_calls(gpu_lib, overlap):
    # D1 = A·Bᵀ, then D2 = D1·Cᵀ reads it, launched back to back on one stream
    # with and without the overlapped (programmatic dependent) launch.  D1 is
    # filled with NaN first, so a second kernel that read D1 before the first
    # finished writing it would produce NaN or wrong values.
    w = si.custom(512, 512, 256, seed=31)
    A, B = w.operands()
    C = si.custom(256, 8, 512, seed=32, dist=si.Dist("uniform", -0.125, 0.125)).operands()[0]  # 256 x 512
    o = gpu_lib.Options(overlap_launch=overlap)
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C)
    for _ in range(4):
        D1 = torch.full((512, 512), float("nan"), dtype=torch.float16, device="cuda")
        gpu_lib.gemm_f16_nt(dA, dB, D1, options=o)
        D2 = gpu_lib.gemm_f16_nt(D1, dC, options=o)
        assert gpu_lib.last_device_status()[0] == 0
        D1h = D1.cpu().numpy()
        assert_close(D1h, oracle.gemm_f16_nt(A, B), "first")
        assert_close(D2.cpu().numpy(), oracle.gemm_f16_nt(D1h, C), "second (reads the first)")


def test_dependent_chain_with_overlap_matches_plain_launches(gpu_lib):
    # A longer chain on CTA-pair kernels: D2 = (A·Bᵀ)·Cᵀ, twenty times over with fresh data.
    # Under the overlapped launch the second GEMM prefetches its first k-tiles of D1 into L2
    # while the first GEMM may still be writing D1; plain launches (overlap_launch = -1)
    # give the reference.  The kernels compute identically either way, so any stale read
    # would show as a bit difference.
    M, N, K, N2 = 2048, 2048, 1024, 1024
    on, off = gpu_lib.Options(overlap_launch=1), gpu_lib.Options(overlap_launch=-1)
    assert gpu_lib.describe(M, N, K, on)["cta_group"] == 2 and gpu_lib.describe(M, N2, N, on)["cta_group"] == 2
    rng = torch.Generator(device="cuda").manual_seed(123)
    outs, refs = [], []
    for _ in range(20):
        dA = (torch.rand((M, K), generator=rng, device="cuda") - 0.5).half()
        dB = (torch.rand((N, K), generator=rng, device="cuda") - 0.5).half()
        dC = ((torch.rand((N2, N), generator=rng, device="cuda") - 0.5) * 0.125).half()
        D1 = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        gpu_lib.gemm_f16_nt(dA, dB, D1, options=on)
        outs.append(gpu_lib.gemm_f16_nt(D1, dC, options=on))
        R1 = gpu_lib.gemm_f16_nt(dA, dB, options=off)
        refs.append(gpu_lib.gemm_f16_nt(R1, dC, options=off))
    torch.cuda.synchronize()
    assert gpu_lib.last_device_status()[0] == 0
    for i, (o, r) in enumerate(zip(outs, refs)):
        assert not torch.isnan(o).any(), f"chain {i}: NaN from a stale read of D1"
        assert torch.equal(o.view(torch.int16), r.view(torch.int16)), f"chain {i} differs"


def test_concurrent_host_threads(gpu_lib):
    # Four host threads, each on its own stream, call the library at once
    # (device set-up is guarded; tensor maps are built per call).  Two of them
    # run K split across thread-block clusters (tiny tiles over 4 CTAs, narrow
    # tiles over 2), whose clusters then share the GPU with the others' grids.
    import threading

    shapes = [(256, 520, 200), (320, 520, 208), (384, 264, 1024), (448, 264, 1088)]
    options = [None, None, gpu_lib.Options(cluster_k=4), gpu_lib.Options(block_m=128, cluster_k=2)]
    assert gpu_lib.describe(*shapes[2], options[2])["cluster_k"] == 4
    assert gpu_lib.describe(*shapes[3], options[3])["cluster_k"] == 2
    probs = [si.custom(M, N, K, seed=60 + t).operands() for t, (M, N, K) in enumerate(shapes)]
    outs = [None] * 4
    errors = []

    def worker(t):
        try:
            A, B = probs[t]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                dA, dB = to_dev(A), to_dev(B)
                for _ in range(10):
                    D = gpu_lib.gemm_f16_nt(dA, dB, stream=s, options=options[t])
            s.synchronize()
            outs[t] = D.cpu().numpy()
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert gpu_lib.last_device_status()[0] == 0
    for (A, B), D in zip(probs, outs):
        assert_close(D, oracle.gemm_f16_nt(A, B), "thread")


def test_repeated_calls_and_streams(gpu_lib):
    w = si.WORKLOADS["ktile_grid_256x256x512"]
    A, B = w.operands()
    ref = oracle.gemm_f16_nt(A, B)
    dA, dB = to_dev(A), to_dev(B)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(5):
            outs.append(gpu_lib.gemm_f16_nt(dA, dB, stream=s))
    s.synchronize()
    assert gpu_lib.last_device_status(s)[0] == 0
    for o in outs:
        assert_close(o.cpu().numpy(), ref, "repeat")


def test_host_pipeline_end_to_end(gpu_lib):
    # Host-buffer path with overlapped copies: three different problems in
    # flight through two device slots; every result must match its own oracle.
    probs = [si.custom(384, 520, 264, seed=s).operands() for s in (41, 42, 43, 44, 45)]
    pipe = gpu_lib.HostPipeline(384, 520, 264)
    outs = [torch.empty((384, 520), dtype=torch.float16).pin_memory() for _ in probs]
    for (A, B), D in zip(probs, outs):
        pipe.submit(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(), D)
    pipe.synchronize()
    assert gpu_lib.last_device_status()[0] == 0
    for (A, B), D in zip(probs, outs):
        assert_close(D.numpy(), oracle.gemm_f16_nt(A, B), "pipeline")
    A, B = probs[0]
    single = gpu_lib.gemm_f16_nt_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory())
    assert_close(single.numpy(), oracle.gemm_f16_nt(A, B), "single host call")


def test_host_buffer_entry_point(gpu_lib):
    # gemm_f16_nt_host through the C ABI: pinned and pageable host operands, the caller's device
    # buffers, copy-in, GEMM and copy-out enqueued on one side stream; D_host must equal the
    # oracle once the stream is done, including the thin, pair and K = 0 paths.
    lib = gpu_lib.load()
    s = torch.cuda.Stream()
    for (M, N, K), pinned in (((128, 128, 64), True), ((300, 520, 200), True), ((1000, 264, 1000), False),
                              ((64, 64, 0), True)):
        A, B = si.custom(M, N, K, seed=M + 2 * N + 3 * K).operands()
        Ah, Bh = torch.from_numpy(A), torch.from_numpy(B)
        Dh = torch.full((M, N), float("nan"), dtype=torch.float16)
        if pinned:
            Ah, Bh, Dh = Ah.pin_memory(), Bh.pin_memory(), Dh.pin_memory()
        dA = torch.empty((M, K), dtype=torch.float16, device="cuda")
        dB = torch.empty((N, K), dtype=torch.float16, device="cuda")
        dD = torch.empty((M, N), dtype=torch.float16, device="cuda")
        rc = lib.gemm_f16_nt_host(Ah.data_ptr() if K else None, Bh.data_ptr() if K else None, Dh.data_ptr(),
                                  M, N, K, dA.data_ptr() if K else None, dB.data_ptr() if K else None,
                                  dD.data_ptr(), s.cuda_stream, None)
        assert rc == 0, gpu_lib.status_string(rc)
        s.synchronize()
        assert gpu_lib.last_device_status(s)[0] == 0
        if K == 0:
            assert not Dh.float().abs().sum().item()
        else:
            assert_close(Dh.numpy(), oracle.gemm_f16_nt(A, B), f"host entry {M}x{N}x{K} pinned={pinned}")


def test_cuda_graph_capture_and_replay(gpu_lib):
    # Launches captured in a CUDA graph (after a first eager call has done the
    # per-device set-up) replay correctly, including a GEMM that reads the
    # previous one's output through the overlapped launch.
    w = si.custom(384, 512, 256, seed=51)
    A, B = w.operands()
    C = si.custom(256, 8, 512, seed=52, dist=si.Dist("uniform", -0.125, 0.125)).operands()[0]
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C)
    D1 = torch.empty((384, 512), dtype=torch.float16, device="cuda")
    D2 = torch.empty((384, 256), dtype=torch.float16, device="cuda")
    gpu_lib.gemm_f16_nt(dA, dB, D1)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        gpu_lib.gemm_f16_nt(dA, dB, D1, stream=s)
        gpu_lib.gemm_f16_nt(D1, dC, D2, stream=s)
    for _ in range(3):
        D1.fill_(float("nan"))
        D2.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert gpu_lib.last_device_status()[0] == 0
        D1h = D1.cpu().numpy()
        assert_close(D1h, oracle.gemm_f16_nt(A, B), "graph first")
        assert_close(D2.cpu().numpy(), oracle.gemm_f16_nt(D1h, C), "graph second")


# ------------------------------------------------------ full-size compares --

def _assert_close_by_rows(got, ref_bits, what, rows_per_chunk=512):
    """assert_close over whole row bands, so that the float64 temporaries stay small."""
    for r0 in range(0, got.shape[0], rows_per_chunk):
        assert_close(got[r0:r0 + rows_per_chunk], ref_bits[r0:r0 + rows_per_chunk], f"{what} rows {r0}..")


@pytest.mark.parametrize("name", ["square_4096", "square_8192", "mlp_proj_8192x28672x4096"])
def test_full_size_workloads_full(gpu_lib, name):
    # The whole of D against the whole of the oracle's D, for the default options (the launch
    # configuration the benchmark times: persistent CTA pairs with one MMA consumer and 256 x 256
    # tiles, or two consumers and 512 x 256 tiles with a long K) and for the other consumer count.  Every 128 x 128 block of D has its owner
    # CTA ("TIRx GEMM detailed technical notes", V8 "Output Ownership"), so a full compare covers
    # every owner, every tile border and the half tiles of the split last wave.
    w = si.WORKLOADS[name]
    A, B = w.operands()
    ref = oracle.gemm_f16_nt(A, B)  # all host threads; about a minute for the largest shape
    default = gpu_lib.describe(w.M, w.N, w.K)["consumers"]
    for options in (None, gpu_lib.Options(consumers=3 - default)):  # the default, then the other count
        D = run(gpu_lib, A, B, options)
        assert np.isfinite(D.astype(np.float32)).all()
        _assert_close_by_rows(D, ref, f"{name} consumers={default if options is None else 3 - default}")
