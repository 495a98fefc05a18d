"""Host-side tests of the C ABI (no GPU needed, no compute call is made).

* the library builds for sm_103a, loads, and exports every entry point that
  include/gemm_f16.h declares;
* argument validation returns its codes before any CUDA work;
* the scheduler, the per-CTA origin and the ring bookkeeping — the same code
  the kernel runs — against the pages' worked examples (tests/golden) and
  against exhaustive properties (bijection, ownership).
"""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import blackwell_tensor_core_02_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")

OK, INVALID, UNSUPPORTED, MISALIGNED, NO_DEVICE = 0, -1, -2, -3, -4


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def declared_functions():
    with open(os.path.join(ROOT, "include", "gemm_f16.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_f16_\w+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 8
    for lib in (g.load(), g.load_checked()):  # the production build and the checked build
        for name in names:
            assert hasattr(lib, name), f"{name} declared in include/gemm_f16.h but not exported"


def test_header_is_c99_and_the_binding_matches_its_layouts():
    """include/gemm_f16.h compiles as strict C99, a C program links against the library and
    calls it, and the ctypes mirrors in the Python binding have the C compiler's sizes and
    field offsets for every struct of the ABI."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    structs = {"gemm_f16_options": g.Options, "gemm_f16_launch_info": g.LaunchInfo,
               "gemm_f16_work_item": g.WorkItem}
    lines = ['#include "gemm_f16.h"', "#include <stddef.h>", "#include <stdio.h>", "int main(void) {",
             '    printf("supported %d\\n", gemm_f16_nt_supported(128, 128, 64));']
    for cname, py in structs.items():
        lines.append(f'    printf("{cname} size %d\\n", (int)sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'    printf("{cname} {field} %d\\n", (int)offsetof({cname}, {field}));')
    lines += ["    return 0;", "}"]
    lib = g.load()  # builds the library if needed
    out_dir = os.path.join(ROOT, "blackwell_tensor_core_02_gb300", "_build", "abi_c_check")
    os.makedirs(out_dir, exist_ok=True)
    src, exe = os.path.join(out_dir, "abi.c"), os.path.join(out_dir, "abi")
    with open(src, "w") as f:
        f.write("\n".join(lines) + "\n")
    lib_dir = os.path.dirname(lib._name)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    src, "-L", lib_dir, "-lgemm_f16", f"-Wl,-rpath,{lib_dir}", "-o", exe], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([exe], check=True, capture_output=True,
                                                              text=True).stdout.splitlines())
    assert got["supported"] == "1"
    for cname, py in structs.items():
        assert int(got[f"{cname} size"]) == ctypes.sizeof(py), cname
        for field, _ in py._fields_:
            assert int(got[f"{cname} {field}"]) == getattr(py, field).offset, (cname, field)


def test_supported_shapes():
    ok = [(128, 128, 64), (4096, 4096, 4096), (8192, 28672, 4096), (1, 8, 8), (0, 8, 8), (5, 0, 0),
          (129, 264, 520), (2 ** 31 - 1024, 8, 8), (8, 2 ** 31 - 1024, 8), (8, 8, 2 ** 31 - 1024)]
    # up to 2^31 - 1024: past that a last tile's coordinates would wrap in 32 bits
    bad = [(128, 12, 64), (128, 128, 60), (-1, 8, 8), (8, 8, -8), (2 ** 31, 8, 8), (8, 2 ** 31, 8),
           (2 ** 31 - 1023, 8, 8), (2 ** 31 - 1, 8, 8), (8, 2 ** 31 - 1016, 8), (8, 8, 2 ** 31 - 1016)]
    for s in ok:
        assert g.gemm_f16_nt_supported(*s), s
    for s in bad:
        assert not g.gemm_f16_nt_supported(*s), s


def test_argument_errors_are_returned_before_any_launch():
    lib = g.load()
    a, b, d = 0x10000, 0x20000, 0x30000  # never dereferenced: every case fails validation first
    assert lib.gemm_f16_nt(a, b, d, -1, 8, 8, None) == INVALID
    assert lib.gemm_f16_nt(a, b, d, 128, 12, 64, None) == UNSUPPORTED
    assert lib.gemm_f16_nt(a, b, d, 128, 128, 60, None) == UNSUPPORTED
    assert lib.gemm_f16_nt(None, b, d, 128, 128, 64, None) == INVALID
    assert lib.gemm_f16_nt(a, None, d, 128, 128, 64, None) == INVALID
    assert lib.gemm_f16_nt(a, b, None, 128, 128, 64, None) == INVALID
    assert lib.gemm_f16_nt(a + 2, b, d, 128, 128, 64, None) == MISALIGNED
    assert lib.gemm_f16_nt(a, b + 8, d, 128, 128, 64, None) == MISALIGNED
    assert lib.gemm_f16_nt(a, b, d + 4, 128, 128, 64, None) == MISALIGNED
    # D may not overlap A or B (A spans 16 KiB from a; B 16 KiB from b)
    assert lib.gemm_f16_nt(a, b, a + 0x3ff0, 128, 128, 64, None) == INVALID
    assert lib.gemm_f16_nt(a, b, b - 0x7ff0, 128, 128, 64, None) == INVALID
    assert lib.gemm_f16_nt(a, a, d, 128, 128, 64, None) != INVALID  # A and B may share memory
    # empty products are accepted and launch nothing, even with null operands
    assert lib.gemm_f16_nt(None, None, None, 0, 128, 64, None) == OK
    assert lib.gemm_f16_nt(None, None, None, 128, 0, 64, None) == OK
    # a workspace of non-zero size must exist; negative sizes are rejected
    assert lib.gemm_f16_nt_ws(a, b, d, 128, 128, 64, None, 4096, None, None) == INVALID
    assert lib.gemm_f16_nt_ws(a, b, d, 128, 128, 64, 0x40000, -1, None, None) == INVALID
    assert lib.gemm_f16_nt_ws(None, None, None, 0, 128, 64, None, 0, None, None) == OK
    for bad in (g.Options(cta_group=3), g.Options(max_clusters=-1), g.Options(raster_group=-2),
                g.Options(debug_flags=2), g.Options(timeout_ns=-5), g.Options(overlap_launch=2),
                g.Options(consumers=3), g.Options(cta_group=1, consumers=2), g.Options(block_n=128),
                g.Options(block_n=32), g.Options(block_n=64, cta_group=2), g.Options(block_n=64, consumers=2),
                g.Options(block_m=32), g.Options(block_m=256), g.Options(block_m=64, block_n=256),
                g.Options(block_m=64, cta_group=2), g.Options(block_m=64, consumers=2),
                g.Options(cluster_k=3), g.Options(cluster_k=16), g.Options(cluster_k=-1),
                g.Options(cluster_k=4, block_n=256),
                g.Options(cluster_k=8, cta_group=2), g.Options(cluster_k=2, consumers=2),
                g.Options(block_n=16, block_m=128), g.Options(block_n=16, cluster_k=2), g.Options(block_n=16, cta_group=2),
                g.Options(block_n=16, consumers=2), g.Options(block_n=8)):
        assert g.gemm_f16_nt_ptr(a, b, d, 128, 128, 64, None, bad) == INVALID


def test_host_buffer_entry_checks_its_arguments_first():
    """gemm_f16_nt_host checks the device buffers as every compute entry point does, and the
    host buffers for null, before it enqueues anything (no GPU needed: every case fails
    validation, and valid arguments then meet the missing device)."""
    lib = g.load()
    h, a, b, d = 0x50000, 0x10000, 0x20000, 0x30000  # never dereferenced
    call = lambda *args: lib.gemm_f16_nt_host(*args, None, None)  # noqa: E731
    assert call(h, h, h, 128, 128, 64, a, b, None) == INVALID          # no device D
    assert call(h, h, h, 128, 128, 64, None, b, d) == INVALID          # no device A
    assert call(h, h, None, 128, 128, 64, a, b, d) == INVALID          # no host D
    assert call(None, h, h, 128, 128, 64, a, b, d) == INVALID          # no host A
    assert call(h, h, h, 128, 128, 64, a + 2, b, d) == MISALIGNED
    assert call(h, h, h, 128, 12, 64, a, b, d) == UNSUPPORTED
    assert call(h, h, h, 128, 128, 64, a, b, a + 0x1000) == INVALID    # device D overlaps device A
    assert call(None, None, None, 0, 128, 64, None, None, None) == OK  # empty product
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert call(h, h, h, 128, 128, 64, a, b, d) == NO_DEVICE


def test_no_device_reported_without_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("only meaningful on a machine without a GPU (the pointers here are fake)")
    lib = g.load()
    assert lib.gemm_f16_nt(0x10000, 0x20000, 0x30000, 128, 128, 64, None) == NO_DEVICE
    assert lib.gemm_f16_nt_workspace_size(256, 256, 4096, None) == NO_DEVICE
    assert lib.gemm_f16_nt_workspace_size(256, 12, 4096, None) == UNSUPPORTED
    info = g.LaunchInfo()
    assert lib.gemm_f16_nt_describe(128, 128, 64, None, 0, ctypes.byref(info)) == NO_DEVICE


def test_describe_validates_before_touching_a_device():
    lib = g.load()
    info = g.LaunchInfo()
    assert lib.gemm_f16_nt_describe(-1, 8, 8, None, 0, ctypes.byref(info)) == INVALID
    assert lib.gemm_f16_nt_describe(128, 12, 64, None, 0, ctypes.byref(info)) == UNSUPPORTED
    assert lib.gemm_f16_nt_describe(128, 128, 64, None, 2, ctypes.byref(info)) == INVALID
    assert lib.gemm_f16_nt_describe(128, 128, 64, None, 0, None) == INVALID
    assert lib.gemm_f16_nt_describe(128, 128, 64, ctypes.byref(g.Options(block_n=64, cta_group=2)), 0,
                                    ctypes.byref(info)) == INVALID
    # an empty product launches no GEMM: all zero, no device needed
    assert g.describe(0, 128, 64) == dict(cta_group=0, consumers=0, block_n=0, split_k=0, block_m=0, stages=0,
                                          clusters=0, work_items=0, workspace_bytes=0, cluster_k=0)


def test_status_strings():
    for code, name in g.STATUS.items():
        assert g.status_string(code).startswith(name)
    assert "unknown" in g.status_string(12345)


@pytest.mark.parametrize("M,N,cg,group,clusters", [
    (4096, 4096, 2, 8, 74), (4096, 4096, 2, 8, 76), (8192, 28672, 2, 8, 76), (4096, 4096, 1, 8, 148),
    (300, 520, 2, 8, 3), (1, 8, 1, 1, 1), (2560, 1280, 2, 3, 7), (1000, 7000, 1, 5, 13), (128, 128, 2, 8, 1),
    (128, 128, 2, 8, 76), (8192, 8192, 2, 8, 76), (1024, 1024, 2, 8, 5),
    (4096, 4096, 4, 8, 76), (8192, 28672, 4, 0, 76), (640, 776, 4, 2, 7),
])
def test_schedule_covers_every_output_once(M, N, cg, group, clusters):
    """Every 128-column block of every tile is computed by exactly one work item.

    cg = 4 stands for a CTA pair with two MMA consumers (512-row tiles).
    """
    consumers = 2 if cg == 4 else 1
    cg = 2 if cg == 4 else cg
    num_m = -(-M // (128 * cg * consumers))
    num_n = -(-N // 256)
    tiles = num_m * num_n
    cover = {}
    per_cluster = []
    for c in range(clusters):
        it = 0
        while True:
            w = g.schedule(M, N, cg, group, clusters, c, it, consumers=consumers)
            if w is None:
                break
            m_idx, n_idx, n_off, n_len = w[:4]
            assert w[4:] == (0, 0, -(-4096 // 64))  # no split-K: every item runs all of K
            assert 0 <= m_idx < num_m and 0 <= n_idx < num_n and n_len in (128, 256)
            for half in range(n_off // 128, (n_off + n_len) // 128):
                key = (m_idx, n_idx, half)
                assert key not in cover, f"{key} computed twice"
                cover[key] = (c, it)
            it += 1
        per_cluster.append(it)
    assert len(cover) == 2 * tiles
    r = tiles % clusters
    split = 0 < 2 * r <= clusters
    items = tiles + (r if split else 0)
    # items are dealt round-robin: cluster c has the items c, c + P, ...
    assert per_cluster == [len(range(c, items, clusters)) for c in range(clusters)]
    # with a split, no cluster runs more than ceil(tiles / P) - 1/2 tile-times
    if split:
        work = [0.0] * clusters
        for (_, _, _), (c, _) in cover.items():
            work[c] += 0.5
        assert max(work) == tiles // clusters + 0.5


def test_default_raster_group_keeps_a_32mib_a_panel():
    # 0 = automatic: the largest group of 256-row M-tiles whose A panel fits 32 MiB.
    def group_of(M, N, K, cg=2):
        first = [g.schedule(M, N, cg, 0, 1, 0, i, K=K)[0] for i in range(40)]
        return next((i for i, m in enumerate(first) if m == 0 and i > 0), None)
    assert group_of(8192, 28672, 4096) == 16  # 16 x 256 rows x 4096 x 2 B = 32 MiB
    assert group_of(8192, 8192, 8192) == 8
    assert group_of(2048, 8192, 4096) == 8    # capped at the 8 M-tiles there are


def test_schedule_grouped_order():
    # 16 x 16 tiles, groups of 8 M-tiles: M fastest inside a group, then N; the second
    # group walks N backwards, starting on the B panels the first one ended on.
    order = [g.schedule(4096, 4096, 2, 8, 1, 0, i)[:2] for i in range(256)]
    assert order[:9] == [(m, 0) for m in range(8)] + [(0, 1)]
    assert order[127] == (7, 15) and order[128] == (8, 15) and order[136] == (8, 14)
    assert order[255] == (15, 0)
    # a ragged last group (5 of 3 + 2 M-tiles) also turns, and every tile comes once
    order = [g.schedule(1280, 1024, 2, 3, 1, 0, i)[:2] for i in range(20)]
    assert order[12:] == [(3, 3), (4, 3), (3, 2), (4, 2), (3, 1), (4, 1), (3, 0), (4, 0)]
    assert sorted(order) == [(m, n) for m in range(5) for n in range(4)]


@pytest.mark.parametrize("M,N,K,cg,clusters,slices", [
    (256, 256, 4096, 2, 76, 8),     # 1 tile: S = min(76, 64/8, 16) = 8
    (1024, 1024, 4096, 2, 76, 4),   # 16 tiles: S = 76 // 16 = 4
    (256, 4096, 2048, 2, 76, 4),    # 16 tiles, 32 K tiles: S = min(4, 4) = 4
    (300, 520, 3000, 2, 76, 5),     # 6 tiles, 47 K tiles: S = 47 // 8 = 5, ragged K slices
    (256, 256, 4096, 1, 152, 8),    # single-CTA tiles
    (1536, 1536, 4096, 2, 76, 1),   # 36 tiles: at most 2 slices would fit, so no split-K
    (256, 256, 512, 2, 76, 1),      # 8 K tiles: too short to split
])
def test_split_k_schedule_covers_k_once(M, N, K, cg, clusters, slices):
    num_m = -(-M // (128 * cg))
    num_n = -(-N // 256)
    k_tiles = -(-K // 64)
    seen = {}
    got_slices = set()
    for c in range(clusters):
        it = 0
        while (w := g.schedule(M, N, cg, 0, clusters, c, it, K=K, split_k=1)) is not None:
            m_idx, n_idx, n_off, n_len, sl, kb, ke = w
            got_slices.add(sl)
            if slices > 1:
                assert (n_off, n_len) == (0, 256) and kb < ke and ke - kb >= 8
            for kt in range(kb, ke):
                for half in range(n_off // 128, (n_off + n_len) // 128):
                    key = (m_idx, n_idx, half, kt)
                    assert key not in seen, f"{key} twice"
                    seen[key] = c
            it += 1
    assert len(seen) == num_m * num_n * 2 * k_tiles
    assert got_slices == set(range(slices))


def test_schedule_splits_the_last_wave_of_4096():
    # 256 tiles over 76 CTA pairs: 3 full waves (228 tiles), then 28 tiles split
    # into 56 half tiles, one per pair, so the tail lasts half a tile.
    items = []
    for c in range(76):
        it = 0
        while (w := g.schedule(4096, 4096, 2, 8, 76, c, it)) is not None:
            items.append((c, it, w))
            it += 1
    assert len(items) == 228 + 56
    assert all(w[3] == 256 for c, it, w in items if it < 3)
    assert all(w[3] == 128 for c, it, w in items if it == 3)
    # split_k does not change a shape with this many tiles
    assert all(g.schedule(4096, 4096, 2, 8, 76, c, it, split_k=1) == w for c, it, w in items)
    assert sum(1 for c, it, w in items if it == 3) == 56


@pytest.mark.parametrize("M,N,K,clusters", [
    (128, 128, 64, 152), (256, 256, 512, 152), (1024, 1024, 512, 152), (300, 520, 256, 7), (1, 8, 8, 1),
    (4096, 4096, 4096, 152), (1000, 7000, 512, 13),
])
def test_narrow_schedule_covers_every_output_once(M, N, K, clusters):
    """Narrow tiles (block_n 64): every 128 x 64 tile is one work item, never split along N or K,
    dealt round-robin over the clusters, also when split-K is asked for."""
    num_m, num_n = -(-M // 128), -(-N // 64)
    k_tiles = -(-K // 64)
    cover = {}
    for c in range(clusters):
        it = 0
        while (w := g.schedule(M, N, 1, 0, clusters, c, it, K=K, block_n=64, split_k=1)) is not None:
            m_idx, n_idx, n_off, n_len, sl, kb, ke = w
            assert (n_off, n_len, sl, kb, ke) == (0, 64, 0, 0, k_tiles)
            assert 0 <= m_idx < num_m and 0 <= n_idx < num_n
            assert (m_idx, n_idx) not in cover
            cover[(m_idx, n_idx)] = c
            it += 1
        assert it == len(range(c, num_m * num_n, clusters))
    assert len(cover) == num_m * num_n
    # cta_group 0 means 1 for narrow tiles; a pair or two consumers are refused
    assert g.schedule(M, N, 0, 0, clusters, 0, 0, K=K, block_n=64) == g.schedule(M, N, 1, 0, clusters, 0, 0, K=K,
                                                                                   block_n=64)
    for cg, consumers in ((2, 1), (2, 2)):
        with pytest.raises(g.GemmError):
            g.schedule(M, N, cg, 0, clusters, 0, 0, K=K, consumers=consumers, block_n=64)
    with pytest.raises(g.GemmError):
        g.schedule(M, N, 1, 0, clusters, 0, 0, K=K, block_n=128)


@pytest.mark.parametrize("M,N,K,clusters", [
    (128, 128, 64, 152), (256, 256, 512, 152), (512, 512, 512, 152), (300, 520, 256, 7), (1, 8, 8, 1),
    (1000, 7000, 512, 13),
])
def test_tiny_schedule_covers_every_output_once(M, N, K, clusters):
    """Tiny tiles (block_m 64, block_n 64): every 64 x 64 tile is one work item, never split along
    N or K, dealt round-robin over the clusters."""
    num_m, num_n = -(-M // 64), -(-N // 64)
    k_tiles = -(-K // 64)
    cover = {}
    for c in range(clusters):
        it = 0
        while (w := g.schedule(M, N, 1, 0, clusters, c, it, K=K, block_n=64, block_m=64, split_k=1)) is not None:
            m_idx, n_idx, n_off, n_len, sl, kb, ke = w
            assert (n_off, n_len, sl, kb, ke) == (0, 64, 0, 0, k_tiles)
            assert 0 <= m_idx < num_m and 0 <= n_idx < num_n
            assert (m_idx, n_idx) not in cover
            cover[(m_idx, n_idx)] = c
            it += 1
        assert it == len(range(c, num_m * num_n, clusters))
    assert len(cover) == num_m * num_n
    # block_n 0 means 64 with block_m 64; block_m 64 needs narrow single-CTA tiles
    assert g.schedule(M, N, 0, 0, clusters, 0, 0, K=K, block_n=0, block_m=64) == \
        g.schedule(M, N, 1, 0, clusters, 0, 0, K=K, block_n=64, block_m=64)
    for kw in (dict(block_n=256), dict(block_n=64, block_m=32), dict(block_n=64, block_m=256)):
        with pytest.raises(g.GemmError):
            g.schedule(M, N, 1, 0, clusters, 0, 0, K=K, **{"block_m": 64, **kw})
    with pytest.raises(g.GemmError):
        g.schedule(M, N, 2, 0, clusters, 0, 0, K=K, block_n=64, block_m=64)


@pytest.mark.parametrize("M,N,K,ks", [
    (256, 256, 512, 4), (256, 256, 512, 8), (128, 128, 128, 2), (200, 72, 4096, 8), (64, 64, 64, 8),
    (64, 64, 192, 8), (1000, 520, 520, 4), (1, 8, 8, 2),
])
@pytest.mark.parametrize("bm", [64, 128])
def test_cluster_k_schedule_covers_every_k_tile_once(M, N, K, ks, bm):
    """Tiny or narrow tiles with K split across clusters (split_k 2, 4, 8 = cluster_k): CTA i of a
    grid of T * S CTAs runs item i, the S consecutive CTAs of tile t take its K slices 0..S-1 in
    order, and S is at most the number of K tiles (halved until it is)."""
    num_m, num_n = -(-M // bm), -(-N // 64)
    k_tiles = -(-K // 64)
    S = ks
    while S > 1 and S > k_tiles:
        S //= 2
    tiles = num_m * num_n
    grid = tiles * S
    seen = {}
    for i in range(grid):
        w = g.schedule(M, N, 1, 0, grid, i, 0, K=K, block_n=64, block_m=bm, split_k=ks)
        assert w is not None
        assert g.schedule(M, N, 1, 0, grid, i, 1, K=K, block_n=64, block_m=bm, split_k=ks) is None
        m_idx, n_idx, n_off, n_len, sl, kb, ke = w
        assert (n_off, n_len, sl) == (0, 64, i % S)
        assert (kb, ke) == (sl * k_tiles // S, (sl + 1) * k_tiles // S) and kb < ke
        seen.setdefault((m_idx, n_idx), []).append((i, kb, ke))
    assert len(seen) == tiles
    for parts in seen.values():
        idx = [i for i, _, _ in parts]
        assert idx == list(range(idx[0], idx[0] + S)) and idx[0] % S == 0  # one cluster per tile
        assert parts[0][1] == 0 and parts[-1][2] == k_tiles
        assert all(parts[j][2] == parts[j + 1][1] for j in range(S - 1))  # contiguous, in slice order
    for bad in (dict(split_k=3), dict(split_k=16), dict(split_k=2, block_n=256, block_m=128)):
        with pytest.raises(g.GemmError):
            g.schedule(M, N, 1, 0, grid, 0, 0, K=K, **{"block_n": 64, "block_m": 64, **bad})


def test_tiny_cta_origin():
    # a 64 x 64 tile: A rows and D rows from m_idx * 64, B rows and D columns from n_idx * 64
    assert g.cta_origin(1, 3, 5, 0, n_len=64, block_n=64, block_m=64) == dict(a_row=192, b_row=320, d_row=192,
                                                                               d_col=320)
    assert g.cta_origin(0, 7, 0, 0, n_len=64, block_n=0, block_m=64) == dict(a_row=448, b_row=0, d_row=448, d_col=0)
    # over a 320 x 192 grid the written 64 x 64 blocks tile D exactly once
    cover = np.zeros((5, 3), dtype=int)
    for m_idx in range(5):
        for n_idx in range(3):
            o = g.cta_origin(1, m_idx, n_idx, 0, n_len=64, block_n=64, block_m=64)
            assert o["a_row"] == o["d_row"] and o["b_row"] == o["d_col"]
            cover[o["d_row"] // 64, o["d_col"] // 64] += 1
    assert np.all(cover == 1)
    for kw in (dict(block_n=256, n_len=256), dict(block_n=64, n_len=64, cta_group=2), dict(block_m=96)):
        args = {"cta_group": 1, "n_len": 64, "block_n": 64, "block_m": 64, **kw}
        with pytest.raises(g.GemmError):
            g.cta_origin(args.pop("cta_group"), 0, 0, 0, **args)


def test_narrow_cta_origin():
    # a 128 x 64 tile: A rows and D rows from m_idx * 128, B rows and D columns from n_idx * 64
    assert g.cta_origin(1, 3, 5, 0, n_len=64, block_n=64) == dict(a_row=384, b_row=320, d_row=384, d_col=320)
    assert g.cta_origin(0, 0, 1, 0, n_len=64, block_n=64) == dict(a_row=0, b_row=64, d_row=0, d_col=64)
    for bad in (dict(n_len=256), dict(n_len=32), dict(n_len=64, n_off=32)):
        with pytest.raises(g.GemmError):
            g.cta_origin(1, 0, 0, 0, block_n=64, **{"n_off": 0, **bad})
    with pytest.raises(g.GemmError):
        g.cta_origin(2, 0, 0, 0, n_len=64, block_n=64)


def test_cta_origin_matches_the_pages_operand_partition():
    for m_idx, n_idx, cbx, a_row, b_row, d_row, d_col in _golden_rows("v8_operand_partition.txt"):
        got = g.cta_origin(2, m_idx, n_idx, cbx)
        assert got == dict(a_row=a_row, b_row=b_row, d_row=d_row, d_col=d_col)
    # a half tile keeps the same partition inside its 128 columns
    assert g.cta_origin(2, 1, 2, 1, n_off=128, n_len=128) == dict(a_row=384, b_row=704, d_row=384, d_col=640)
    assert g.cta_origin(1, 1, 2, 0, n_off=128, n_len=128) == dict(a_row=128, b_row=640, d_row=128, d_col=640)
    # two consumers (TIRx notes V9): the tile is 512 rows; consumer 1's block of
    # each CTA lies 256 rows below consumer 0's, B is shared
    assert g.cta_origin(2, 1, 2, 1, consumers=2) == dict(a_row=640, b_row=640, d_row=640, d_col=512)
    with pytest.raises(g.GemmError):
        g.cta_origin(1, 0, 0, 0, consumers=2)


def test_cta_origin_ownership_covers_each_output_once():
    # Over all tiles and both CTAs, the written 128-row x 256-column blocks tile D exactly once.
    for cg in (1, 2):
        M, N = 1024, 768
        cover = np.zeros((M // 128, N // 256), dtype=int)
        for m_idx in range(M // (128 * cg)):
            for n_idx in range(N // 256):
                for r in range(cg):
                    o = g.cta_origin(cg, m_idx, n_idx, r)
                    assert o["d_row"] == o["a_row"] and o["d_col"] == n_idx * 256
                    cover[o["d_row"] // 128, o["d_col"] // 256] += 1
                    # the B slice loaded by this CTA lies inside the tile's 256 output columns
                    assert n_idx * 256 <= o["b_row"] < (n_idx + 1) * 256
        assert np.all(cover == 1)
    with pytest.raises(g.GemmError):
        g.cta_origin(2, 0, 0, 2)
    with pytest.raises(g.GemmError):
        g.cta_origin(2, 0, 0, 0, n_off=128, n_len=256)


def test_pipeline_state_matches_the_pages_table():
    want = [(s, p) for _, s, p in _golden_rows("v5_stage_phase_depth2.txt")]
    assert g.pipeline_trace(2, 0, 4) == want
    # the producer end runs the same sequence one phase apart
    assert g.pipeline_trace(2, 1, 4) == [(s, 1 - p) for s, p in want]
    # deeper rings: the phase flips exactly when the stage wraps
    tr = g.pipeline_trace(6, 0, 20)
    for i, (s, p) in enumerate(tr):
        assert s == i % 6 and p == (i // 6) % 2
    with pytest.raises(g.GemmError):
        g.pipeline_trace(0, 0, 1)


def _simulate_ring(depth, producer_phase, steps, seed, traces=None):
    """Model one SMEM ring with parity barriers, driven by the library's PipelineState traces
    (or by the given (producer, consumer) traces).

    try_wait(bar, p) passes when the barrier's phase bit differs from p
    ("GEMM I", the phase-flip table).  A fill completes full[s]'s phase; a
    consume completes empty[s]'s phase.  Returns the consumed sequence, or None
    on deadlock.
    """
    if traces is None:
        prod = g.pipeline_trace(depth, producer_phase, steps)
        cons = g.pipeline_trace(depth, 0, steps)
    else:
        prod, cons = traces
    full, empty = [0] * depth, [0] * depth
    slot = [None] * depth
    i = j = 0
    out = []
    rng = random.Random(seed)
    while j < steps:
        can_p = i < steps and empty[prod[i][0]] != prod[i][1]
        can_c = full[cons[j][0]] != cons[j][1]
        if not (can_p or can_c):
            return None
        if can_p and (not can_c or rng.random() < 0.5):
            s = prod[i][0]
            slot[s] = i
            full[s] ^= 1
            i += 1
        else:
            s = cons[j][0]
            out.append(slot[s])
            empty[s] ^= 1
            j += 1
    return out


def test_opposite_initial_phases_model():
    for depth in (1, 2, 4, 6):
        for seed in range(20):
            assert _simulate_ring(depth, 1, 50, seed) == list(range(50))
    # the pages' "subtlest bug": both ends at phase 0 deadlock on the fresh barrier
    assert _simulate_ring(4, 0, 50, 0) is None


def test_forgotten_phase_toggle_corrupts_silently():
    """The pages' other ring bug ("GEMM I", the phase-flip table): a PipelineState that wraps
    its stage but never flips its phase.  Planted in the model, not in a kernel.  After the
    first lap a wait compares against a phase bit that a later fill or drain may already have
    flipped back, so depending on the interleaving the ring either stalls or, worse, runs to
    the end with the consumer reading slots that hold other fills than the ones it expects
    (e.g. fills 0-3 twice, never 4-7).  No interleaving delivers the right data."""
    depth, steps = 4, 40
    stuck = lambda phase: [(i % depth, phase) for i in range(steps)]  # noqa: E731
    silent = 0
    for seed in range(40):
        out = _simulate_ring(depth, 1, steps, seed, traces=(stuck(1), stuck(0)))
        assert out != list(range(steps))
        silent += out is not None
    assert silent > 0, "some interleavings finish with wrong data and nothing to notice it by"
    # the library's traces, same seeds: always in order
    for seed in range(40):
        assert _simulate_ring(depth, 1, steps, seed) == list(range(steps))


# ------------------------------------------- configuration choice, host only --
# gemm_f16_nt_describe_for runs the library's configuration choice for a device
# given by its co-resident cluster counts, without a GPU.  GB300: 152 SMs, one
# CTA of any configuration per SM, so 152 single CTAs, 76 pairs, 36 clusters of
# 4 and 15 of 8 (the GPU test checks these counts on the device itself).
GB300 = [152, 76, 76, 152, 152, 76, 36, 15, 76, 36, 15]
HALF = [76, 38, 38, 76, 76, 38, 18, 7, 38, 18, 7]      # a device with half the SMs
NO_SPLIT = GB300[:5] + [0] * 6                         # one that cannot co-schedule clusters


def test_describe_for_the_five_workloads_on_gb300():
    expect = {
        # thin 64 x 16 tiles: 2 x 8 and 4 x 16 of them, one per CTA, no K split
        (128, 128, 64): dict(cta_group=1, consumers=1, block_n=16, block_m=64, cluster_k=1, clusters=16,
                             work_items=16),
        (256, 256, 512): dict(cta_group=1, consumers=1, block_n=16, block_m=64, cluster_k=1, clusters=64,
                              work_items=64),
        (4096, 4096, 4096): dict(cta_group=2, consumers=1, block_n=256, block_m=128, cluster_k=1, clusters=76,
                                 work_items=284),
        # K = 8192: two consumers, 512 x 256 tiles (16 x 32 = 512 on 76 pairs; the last wave is
        # 56 tiles, more than half of 76, so nothing is split)
        (8192, 8192, 8192): dict(cta_group=2, consumers=2, block_n=256, block_m=128, cluster_k=1, clusters=76,
                                 work_items=512),
        (8192, 28672, 4096): dict(cta_group=2, consumers=1, block_n=256, block_m=128, cluster_k=1, clusters=76,
                                  work_items=3596),
    }
    for (M, N, K), want in expect.items():
        got = g.describe_for(M, N, K, GB300)
        assert {k: got[k] for k in want} == want, (M, N, K)
        assert got["split_k"] == 1 and got["workspace_bytes"] == 0


@pytest.mark.parametrize("M,N,K,consumers", [
    (4096, 4096, 8192, 2), (6144, 6144, 6144, 2), (8192, 8192, 8192, 2), (12288, 12288, 12288, 2),
    (8192, 8192, 16384, 2), (16384, 8192, 8192, 2),
    (4096, 4096, 4096, 1), (8192, 8192, 4096, 1), (8192, 28672, 4096, 1), (8192, 8192, 2048, 1),
    (3072, 3072, 3072, 1),
    # 96 K tiles but 4 x 8 = 32 two-consumer tiles, fewer than one wave of 76 pairs
    (2048, 2048, 6144, 1),
])
def test_describe_for_the_consumer_count_rule(M, N, K, consumers):
    """Two MMA consumers from 96 K tiles of 64 on, when their 512 x 256 tiles fill a wave of
    pairs; given options are kept."""
    c = g.describe_for(M, N, K, GB300)
    assert (c["cta_group"], c["consumers"], c["block_n"], c["split_k"]) == (2, consumers, 256, 1)
    assert c["work_items"] >= -(-M // (256 * consumers)) * -(-N // 256)
    assert g.describe_for(M, N, K, GB300, g.Options(consumers=1))["consumers"] == 1
    assert g.describe_for(M, N, K, GB300, g.Options(consumers=2))["consumers"] == 2
    single = g.describe_for(M, N, K, GB300, g.Options(cta_group=1))
    assert (single["cta_group"], single["consumers"]) == (1, 1)
    # a grid capped below the tile count still counts as a full wave
    assert g.describe_for(M, N, K, GB300, g.Options(max_clusters=8))["consumers"] == (2 if K >= 6144 else 1)


@pytest.mark.parametrize("M,N,K,bm,ks", [
    (256, 256, 4096, 64, 4), (128, 128, 4096, 64, 8), (256, 256, 1024, 64, 4), (128, 1024, 1024, 64, 2),
    (512, 512, 4096, 128, 4), (512, 512, 512, 64, 1), (512, 512, 1024, 64, 1), (576, 576, 1024, 64, 1),
    (640, 640, 4096, 128, 2), (768, 512, 4096, 128, 2), (512, 1024, 4096, 128, 2), (768, 768, 4096, 128, 2),
    (768, 768, 2048, 128, 1), (384, 384, 2048, 128, 4), (512, 512, 2048, 128, 2),
    # tiny tiles: no split below 12 K tiles; clusters of 8 only within a quarter of the CTAs
    (384, 384, 640, 64, 1), (256, 256, 896, 64, 4), (128, 128, 1024, 64, 8), (128, 256, 1024, 64, 4),
    (192, 192, 1024, 64, 4),
])
def test_describe_for_the_cluster_k_split_rule(M, N, K, bm, ks):
    c = g.describe_for(M, N, K, GB300)
    tiles = -(-M // bm) * -(-N // 64)
    assert (c["block_n"], c["block_m"], c["cluster_k"], c["split_k"]) == (64, bm, ks, 1)
    assert (c["clusters"], c["work_items"], c["workspace_bytes"]) == (tiles, tiles * ks, 0)
    # with a workspace the split still wins; without the device's clusters it is off
    assert g.describe_for(M, N, K, GB300, with_workspace=True)["workspace_bytes"] == 0
    assert g.describe_for(M, N, K, NO_SPLIT)["cluster_k"] == 1


@pytest.mark.parametrize("M,N,K,thin", [
    (128, 128, 64, True), (256, 256, 512, True), (128, 128, 512, True), (256, 256, 448, True),
    (128, 256, 256, True), (1, 8, 8, True), (256, 256, 576, True), (256, 256, 768, True),  # up to 12 K tiles
    (256, 256, 832, False),   # 13 K tiles: the cluster K split instead
    (320, 256, 512, False),   # 5 x 16 = 80 thin tiles: more than half a wave, tiny tiles
    (384, 384, 256, False),   # 6 x 24 = 144 thin tiles
    (512, 512, 512, False),   # 8 x 32 = 256 thin tiles: more than a wave
    (1024, 1024, 512, False),  # narrow tiles
])
def test_describe_for_the_thin_tile_rule(M, N, K, thin):
    """Thin 64 x 16 tiles where the tiny tiles would run a K-loop of at most 12 tiles of 64 and
    the thin tiles fill at most half of the co-resident CTAs; only when block_n, block_m and
    cluster_k are all left open."""
    c = g.describe_for(M, N, K, GB300)
    if thin:
        tiles = -(-M // 64) * -(-N // 16)
        assert (c["cta_group"], c["block_n"], c["block_m"], c["cluster_k"], c["split_k"]) == (1, 16, 64, 1, 1)
        assert (c["clusters"], c["work_items"], c["workspace_bytes"], c["stages"]) == (tiles, tiles, 0, 12)
        # any tile option given by the caller keeps the earlier rules
        for o in (g.Options(block_m=64), g.Options(block_n=64), g.Options(cluster_k=1)):
            assert g.describe_for(M, N, K, GB300, o)["block_n"] == 64
        # a grid capped below the thin tile count keeps the tiny tiles
        assert g.describe_for(M, N, K, GB300, g.Options(max_clusters=tiles - 1))["block_n"] in (64, 16 if tiles == 1 else 64)
    else:
        assert c["block_n"] != 16
    forced = g.describe_for(512, 512, 4096, GB300, g.Options(block_n=16))
    assert (forced["block_n"], forced["block_m"], forced["cluster_k"], forced["work_items"]) == (16, 64, 1, 256)


def test_describe_for_the_workspace_split_k_choice():
    capped = g.Options(max_clusters=76)  # a capped grid turns the cluster split off
    deep = g.describe_for(768, 640, 4096, GB300, capped, with_workspace=True)
    assert (deep["cta_group"], deep["block_n"], deep["split_k"], deep["workspace_bytes"]) == (2, 256, 8, 8 * 768 * 640 * 4)
    assert g.describe_for(768, 640, 4096, GB300, with_workspace=True)["workspace_bytes"] == 0
    # 4 slices only: narrow tiles instead
    assert g.describe_for(1024, 1024, 4096, GB300, with_workspace=True)["block_n"] == 64


def test_describe_for_rejects_bad_devices_and_arguments():
    lib = g.load()
    info = g.LaunchInfo()
    counts = (ctypes.c_int32 * 11)(*GB300)
    assert lib.gemm_f16_nt_describe_for(128, 128, 64, None, 0, counts, 10, ctypes.byref(info)) == INVALID
    assert lib.gemm_f16_nt_describe_for(128, 128, 64, None, 0, None, 11, ctypes.byref(info)) == INVALID
    assert lib.gemm_f16_nt_describe_for(128, 128, 64, None, 0, counts, 11, None) == INVALID
    assert lib.gemm_f16_nt_describe_for(128, 128, 64, None, 2, counts, 11, ctypes.byref(info)) == INVALID
    assert lib.gemm_f16_nt_describe_for(128, 12, 64, None, 0, counts, 11, ctypes.byref(info)) == UNSUPPORTED
    for bad in ([0] + GB300[1:], GB300[:4] + [0] + GB300[5:], GB300[:7] + [-1] + GB300[8:]):
        with pytest.raises(g.GemmError):
            g.describe_for(128, 128, 64, bad)
    assert g.describe_for(0, 128, 64, GB300)["clusters"] == 0
    with pytest.raises(g.GemmError):
        g.describe_for(128, 128, 64, GB300, g.Options(cluster_k=3))


@pytest.mark.parametrize("device", [GB300, HALF, NO_SPLIT], ids=["gb300", "half", "no-split"])
def test_describe_for_random_shapes_keep_the_launch_rules(device):
    """Whatever the shape, the chosen configuration respects the launch rules: a K split only
    on 64-wide tiles, one cluster per tile, every cluster co-resident at once, at least one K
    tile per CTA, and no split on a device that cannot run its clusters."""
    rng = np.random.default_rng(5)
    slots = {(64, 2): 5, (64, 4): 6, (64, 8): 7, (128, 2): 8, (128, 4): 9, (128, 8): 10}
    for _ in range(400):
        M = int(rng.integers(1, 6000))
        N = int(rng.integers(1, 800)) * 8
        K = int(rng.choice([int(rng.integers(1, 64)) * 8, int(rng.integers(64, 1200)) * 8]))
        ws = bool(rng.integers(0, 2))
        c = g.describe_for(M, N, K, device, with_workspace=ws)
        k_tiles = -(-K // 64)
        assert c["cluster_k"] in (1, 2, 4, 8) and c["split_k"] >= 1
        if c["block_n"] == 64:
            assert c["cta_group"] == 1 and c["block_m"] in (64, 128) and c["workspace_bytes"] == 0
            tiles = -(-M // c["block_m"]) * -(-N // 64)
        if c["block_n"] == 16:  # thin tiles: short K, one wave, no split
            tiles = -(-M // 64) * -(-N // 16)
            assert (c["cta_group"], c["block_m"], c["cluster_k"], c["split_k"], c["workspace_bytes"]) == (1, 64, 1, 1, 0)
            assert k_tiles <= 12 and 2 * tiles <= device[4] and c["work_items"] == tiles == c["clusters"]
        if c["cluster_k"] > 1:
            assert c["block_n"] == 64 and c["split_k"] == 1
            assert c["clusters"] == tiles and c["work_items"] == tiles * c["cluster_k"]
            assert c["clusters"] <= device[slots[(c["block_m"], c["cluster_k"])]]
            assert c["cluster_k"] <= k_tiles and k_tiles >= (12 if c["block_m"] == 64 else 8)
        elif c["block_n"] == 64:
            assert c["work_items"] == tiles
        if c["split_k"] > 1:
            assert ws and c["block_n"] == 256 and c["workspace_bytes"] == c["split_k"] * M * N * 4
        if device is NO_SPLIT:
            assert c["cluster_k"] == 1


def test_status_codes_are_pinned():
    """The status numbering is part of the ABI: the header's enum, the binding's table and the
    library's status strings agree, and the values stay what they are.  The first eight follow
    the boundary's original list; GEMM_ERR_CUDA (-8) was added for runtime errors that are not a
    launch failure, so the device range-check code moved to -10, and the fixed-scratch refusal
    took -9."""
    with open(os.path.join(ROOT, "include", "gemm_f16.h")) as f:
        text = f.read()
    body = re.search(r"typedef enum gemm_status \{(.*?)\} gemm_status_t;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    header = {name: int(val) for name, val in re.findall(r"(GEMM_\w+)\s*=\s*(-?\d+)", body)}
    expected = {"GEMM_OK": 0, "GEMM_ERR_INVALID_ARG": -1, "GEMM_ERR_UNSUPPORTED_SHAPE": -2,
                "GEMM_ERR_MISALIGNED": -3, "GEMM_ERR_NO_DEVICE": -4, "GEMM_ERR_ARCH": -5, "GEMM_ERR_LAUNCH": -6,
                "GEMM_ERR_DEVICE_TIMEOUT": -7, "GEMM_ERR_CUDA": -8, "GEMM_ERR_SCRATCH_LIMIT": -9,
                "GEMM_ERR_DEVICE_BOUNDS": -10}
    assert header == expected
    assert {name: code for code, name in g.STATUS.items()} == expected
    for name, code in expected.items():
        assert g.status_string(code).split(":")[0] == name
    assert g.status_string(-11) == "unknown gemm_f16 status"


def test_last_device_status_reports_where_through_an_out_parameter():
    """gemm_f16_last_device_status(stream, info) takes an optional uint64_t* beside the stream
    (the boundary's first sketch had the stream alone): NULL is allowed, and without a device
    the call reports GEMM_ERR_NO_DEVICE before touching it."""
    assert "int gemm_f16_last_device_status(void *stream, uint64_t *info);" in open(
        os.path.join(ROOT, "include", "gemm_f16.h")).read()
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("only meaningful on a machine without a GPU")
    lib = g.load()
    info = ctypes.c_uint64(0x1234)
    assert lib.gemm_f16_last_device_status(None, None) == NO_DEVICE
    assert lib.gemm_f16_last_device_status(None, ctypes.byref(info)) == NO_DEVICE
    assert info.value == 0x1234  # untouched on an error before the synchronisation
