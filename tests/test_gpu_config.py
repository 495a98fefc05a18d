"""Which kernel configuration a call resolves to on a GB300 (gemm_f16_nt_describe).

The choices are host logic, but they depend on how many CTAs and CTA pairs are
co-resident on the device, so they are checked here, on the GPU, for the five
workloads and the boundaries between configurations.  Each configuration's
results are checked against the oracle elsewhere; these tests pin which one
runs.
"""
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _resident_tiny_ctas(gpu_lib):
    # a grid of 64 x 64 tiles far beyond one wave launches every co-resident CTA
    return gpu_lib.describe(4096, 4096, 64, gpu_lib.Options(block_m=64))["clusters"]


def test_smallest_problems_take_thin_or_tiny_tiles(gpu_lib):
    # the two small workloads: thin 64 x 16 tiles, one per CTA (K at most 768, half a wave)
    c1 = gpu_lib.describe(128, 128, 64)
    assert (c1["cta_group"], c1["block_n"], c1["block_m"], c1["split_k"], c1["cluster_k"], c1["clusters"],
            c1["work_items"], c1["stages"]) == (1, 16, 64, 1, 1, 16, 16, 12)
    c2 = gpu_lib.describe(256, 256, 512)
    assert (c2["cta_group"], c2["block_n"], c2["block_m"], c2["split_k"], c2["cluster_k"], c2["clusters"],
            c2["work_items"]) == (1, 16, 64, 1, 1, 64, 64)
    for M, N, K in ((128, 128, 512), (256, 256, 448), (128, 256, 256), (256, 256, 768)):  # thin tiles as well
        c = gpu_lib.describe(M, N, K)
        tiles = -(-M // 64) * -(-N // 16)
        assert (c["block_n"], c["block_m"], c["cluster_k"], c["work_items"], c["clusters"]) == \
            (16, 64, 1, tiles, tiles), (M, N, K)
    # 64 x 64 tiles up to two thirds of the co-resident CTAs, any K, without a workspace
    P = _resident_tiny_ctas(gpu_lib)
    assert P >= 140  # GB300: 152 SMs, one tiny-tile CTA each
    for M, N, K in ((512, 512, 512), (64 * (2 * P // 3), 64, 1024), (576, 576, 1024), (200, 1000, 72)):
        c = gpu_lib.describe(M, N, K)
        tiles = -(-M // 64) * -(-N // 64)
        assert (c["block_n"], c["block_m"], c["cluster_k"], c["work_items"], c["clusters"]) == \
            (64, 64, 1, tiles, tiles), (M, N, K)
        assert c["workspace_bytes"] == 0


def test_long_k_on_few_tiles_splits_k_across_clusters(gpu_lib):
    # from 8 K tiles of 64 on (12 for tiny tiles), 64-wide tiles split K across a cluster: the
    # largest of 8, 4, 2 CTAs that leaves each at least 2 K tiles, with tiles * cluster_k at most
    # half the co-resident CTAs (a quarter for tiny tiles in clusters of 8; a whole wave with at
    # least 24 K tiles per CTA); narrow tiles instead of tiny ones
    # where the tiny ones get no split but the narrow ones do with at least 16 K tiles per CTA,
    # or where the tiny ones split in 2 and the narrow ones can split in 4 with at least 8
    for (M, N, K), bm, ks in (((256, 256, 4096), 64, 4), ((128, 128, 4096), 64, 8), ((256, 256, 1024), 64, 4),
                              ((128, 1024, 1024), 64, 2), ((384, 384, 2048), 128, 4), ((512, 512, 4096), 128, 4),
                              ((512, 512, 512), 64, 1), ((512, 512, 1024), 64, 1), ((576, 576, 1024), 64, 1),
                              ((640, 640, 4096), 128, 2), ((768, 512, 4096), 128, 2), ((512, 1024, 4096), 128, 2),
                              ((768, 768, 4096), 128, 2), ((768, 768, 2048), 128, 1), ((512, 512, 2048), 128, 2),
                              ((384, 384, 640), 64, 1), ((256, 256, 896), 64, 4), ((128, 256, 1024), 64, 4)):
        c = gpu_lib.describe(M, N, K)
        tiles = -(-M // bm) * -(-N // 64)
        assert (c["block_n"], c["block_m"], c["cluster_k"], c["split_k"]) == (64, bm, ks, 1), (M, N, K)
        assert (c["clusters"], c["work_items"], c["workspace_bytes"]) == (tiles, tiles * ks, 0), (M, N, K)
        # it needs no workspace, and wins over split-K through one
        w = gpu_lib.describe(M, N, K, with_workspace=True)
        if ks > 1:
            assert (w["block_m"], w["cluster_k"], w["workspace_bytes"]) == (bm, ks, 0), (M, N, K)
            assert gpu_lib.workspace_size(M, N, K) == 0
    # forced: at most one CTA per K tile; off; and not with a capped persistent grid
    assert gpu_lib.describe(256, 256, 512, gpu_lib.Options(cluster_k=8))["cluster_k"] == 8
    assert gpu_lib.describe(256, 256, 128, gpu_lib.Options(cluster_k=8))["cluster_k"] == 2
    assert gpu_lib.describe(256, 256, 64, gpu_lib.Options(cluster_k=4))["cluster_k"] == 1
    assert gpu_lib.describe(256, 256, 4096, gpu_lib.Options(cluster_k=1))["cluster_k"] == 1
    assert gpu_lib.describe(256, 256, 4096, gpu_lib.Options(max_clusters=5))["cluster_k"] == 1
    forced = gpu_lib.describe(1000, 520, 1000, gpu_lib.Options(cluster_k=4))  # more clusters than fit at once
    assert (forced["block_m"], forced["cluster_k"], forced["clusters"]) == (64, 4, 16 * 9)
    narrow = gpu_lib.describe(1000, 520, 1000, gpu_lib.Options(cluster_k=4, block_m=128))
    assert (narrow["block_n"], narrow["block_m"], narrow["cluster_k"], narrow["clusters"], narrow["stages"]) == \
        (64, 128, 4, 8 * 9, 8)


def test_small_problems_take_narrow_tiles(gpu_lib):
    P = _resident_tiny_ctas(gpu_lib)
    # one wave of 128 x 64 tiles, but more than two thirds of a wave of 64 x 64 tiles
    for M, N, K in ((1024, 1024, 1024), (1024, 1024, 4096), (128, 4096, 2048), (64 * (2 * P // 3 + 1), 64, 1024)):
        c = gpu_lib.describe(M, N, K)
        assert (c["block_n"], c["block_m"], c["stages"]) == (64, 128, 8), (M, N, K)
        assert c["work_items"] == -(-M // 128) * -(-N // 64), (M, N, K)
        assert c["clusters"] == c["work_items"] and c["workspace_bytes"] == 0


def test_more_than_one_wave_keeps_256_wide_tiles(gpu_lib):
    wide = gpu_lib.describe(2048, 1024, 512)  # 256 narrow tiles: more than one wave
    assert (wide["cta_group"], wide["block_n"]) == (1, 256)
    big = gpu_lib.describe(4096, 4096, 4096)
    assert (big["cta_group"], big["consumers"], big["block_n"], big["block_m"], big["split_k"],
            big["stages"]) == (2, 1, 256, 128, 1, 6)
    P, T = big["clusters"], 256
    r = T % P
    assert big["work_items"] == (T + r if 0 < 2 * r <= P else T)
    assert big["clusters"] >= 70  # GB300: 152 SMs, 76 co-resident pairs


def test_split_k_wins_only_with_at_least_8_slices(gpu_lib):
    # Where a K split across clusters applies it wins (checked above); with the grid capped
    # (max_clusters, which also turns the cluster split off) the choice is between narrow
    # tiles and split-K through a workspace: 9 pair tiles with 64 K tiles split 8 ways.
    pairs = gpu_lib.describe(4096, 4096, 4096)["clusters"]
    capped = gpu_lib.Options(max_clusters=pairs)
    deep = gpu_lib.describe(768, 640, 4096, capped, with_workspace=True)
    assert (deep["cta_group"], deep["block_n"], deep["split_k"], deep["cluster_k"]) == (2, 256, 8, 1)
    assert deep["workspace_bytes"] == 8 * 768 * 640 * 4 == gpu_lib.workspace_size(768, 640, 4096, capped)
    assert gpu_lib.workspace_size(768, 640, 4096) == 0  # by default the narrow tiles split K in clusters
    shallow = gpu_lib.describe(1024, 1024, 4096, with_workspace=True)  # 4 slices: narrow tiles instead
    assert shallow["block_n"] == 64 and shallow["split_k"] == 1 and gpu_lib.workspace_size(1024, 1024, 4096) == 0
    tiny = gpu_lib.describe(256, 256, 1024, with_workspace=True)  # split-K would give 2 slices: tiny tiles
    assert (tiny["block_m"], tiny["split_k"]) == (64, 1)


def test_explicit_options_are_obeyed(gpu_lib):
    single = gpu_lib.describe(128, 128, 64, gpu_lib.Options(cta_group=1))
    assert (single["cta_group"], single["block_n"]) == (1, 256)
    pair = gpu_lib.describe(128, 128, 64, gpu_lib.Options(cta_group=2))
    assert (pair["cta_group"], pair["block_n"]) == (2, 256)
    two = gpu_lib.describe(4096, 4096, 4096, gpu_lib.Options(consumers=2))
    assert (two["cta_group"], two["consumers"], two["block_n"]) == (2, 2, 256)
    narrow = gpu_lib.describe(4096, 4096, 4096, gpu_lib.Options(block_n=64))
    assert (narrow["cta_group"], narrow["block_n"], narrow["block_m"], narrow["work_items"]) == (1, 64, 128, 32 * 64)
    forced = gpu_lib.describe(128, 128, 64, gpu_lib.Options(block_m=128))
    assert (forced["block_n"], forced["block_m"], forced["work_items"]) == (64, 128, 2)
    tiny = gpu_lib.describe(4096, 4096, 4096, gpu_lib.Options(block_m=64))
    assert (tiny["cta_group"], tiny["block_n"], tiny["block_m"], tiny["work_items"]) == (1, 64, 64, 64 * 64)
    capped = gpu_lib.describe(4096, 4096, 4096, gpu_lib.Options(max_clusters=5))
    assert capped["clusters"] == 5


def test_host_query_agrees_with_the_device(gpu_lib):
    # The device's own co-resident counts are the fixture the host-only tests use, and the
    # host-only query with them gives what the device query gives, for any shape and options.
    import numpy as np

    counts = gpu_lib.co_resident()
    assert counts == [152, 76, 76, 152, 152, 76, 36, 15, 76, 36, 15]
    rng = np.random.default_rng(9)
    opts = [None, gpu_lib.Options(cta_group=1), gpu_lib.Options(block_m=64), gpu_lib.Options(block_m=128, block_n=64),
            gpu_lib.Options(cluster_k=4), gpu_lib.Options(max_clusters=7), gpu_lib.Options(consumers=2)]
    for _ in range(300):
        M = int(rng.integers(1, 9000))
        N = int(rng.integers(1, 1200)) * 8
        K = int(rng.integers(1, 1100)) * 8
        o = opts[int(rng.integers(0, len(opts)))]
        ws = bool(rng.integers(0, 2))
        assert gpu_lib.describe(M, N, K, o, with_workspace=ws) == gpu_lib.describe_for(M, N, K, counts, o,
                                                                                        with_workspace=ws), (M, N, K)
