// schedule.h -- ring bookkeeping and the persistent tile scheduler.
//
// Plain integer logic shared by the kernel and by the host queries of the C
// ABI (gemm_f16_nt_schedule, gemm_f16_pipeline_trace), so that the host tests
// exercise exactly what the device runs.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define GEMM_HD __host__ __device__ __forceinline__
#else
#define GEMM_HD inline
#endif

namespace gemm_f16 {

// Stage index and phase bit of one producer-consumer ring ("GEMM III",
// "Four barriers = two producer-consumer rings": PipelineState with .stage,
// .phase and .advance()).  advance() moves to the next buffer and flips the
// phase when the stage index wraps (TIRx notes V5, "Barrier Phase Tracking").
// The producer end starts at phase 1 so that its first wait on a fresh
// barrier passes; the consumer end starts at phase 0 so that it blocks until
// the first fill completes ("The subtlest bug: opposite initial phases").
struct PipelineState {
    int32_t depth;
    int32_t stage;
    uint32_t phase;
    GEMM_HD PipelineState(int32_t depth_, uint32_t phase_) : depth(depth_), stage(0), phase(phase_) {}
    GEMM_HD void advance() {
        if (++stage == depth) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

struct TileCoord {
    int32_t m_idx;
    int32_t n_idx;
};

// Linear tile index -> (m_idx, n_idx) in groups of `group` M-tiles: inside a
// group M varies fastest, then N; groups follow one another along M (TIRx
// notes V6, "Better L2 Locality", l2_group_size = 8).  Odd groups walk N
// backwards (a serpentine, not on the pages), so a group starts on the B
// panels the group before it ended on, while they are still in L2: measured
// on GB300 (ncu, one launch), 8192^3 with two consumers reads 812 MB of DRAM
// instead of 871, 8192x28672x4096 676 instead of 687.  A bijection from
// [0, num_m * num_n) onto the tile grid.
GEMM_HD TileCoord tile_of(int32_t t, int32_t num_m, int32_t num_n, int32_t group) {
    const int32_t per_group = group * num_n;
    const int32_t g = t / per_group;
    const int32_t first_m = g * group;
    const int32_t rest = num_m - first_m;
    const int32_t gsize = rest < group ? rest : group;
    const int32_t r = t - g * per_group;
    TileCoord c;
    c.m_idx = first_m + r % gsize;
    c.n_idx = (g & 1) ? num_n - 1 - r / gsize : r / gsize;
    return c;
}

// Default size of the grouped raster, in M-tiles.  Inside a group the A panel
// (group x tile_m rows x K) is reused by every N-tile while B streams past, so
// B is read from memory once per group: total reads ~ A + ceil(num_m/group)*B.
// Larger groups read less, until the panel no longer stays in L2; the group
// is the largest whose A panel fits in 32 MiB (a quarter of GB300's L2), at
// least 1 and at most num_m.  (TIRx notes V6 fixes l2_group_size = 8 for
// 128x128 tiles at K = 4096, i.e. a 8 MiB panel; the measured optimum on
// GB300 with 256-row tiles is 16 at K = 4096 and 8 at K = 8192, both 32 MiB.)
GEMM_HD int32_t auto_raster_group(int32_t num_m, int64_t K, int32_t tile_m) {
    const int64_t panel = static_cast<int64_t>(tile_m) * (K > 0 ? K : 1) * 2;
    int64_t g = (int64_t(32) << 20) / panel;
    if (g < 1) g = 1;
    if (g > num_m) g = num_m;
    return static_cast<int32_t>(g);
}

// One unit of work of a persistent cluster: a whole tile, or one half of a
// tile split along N.  Splitting the tiles of a last, partly filled wave in
// two lets twice as many clusters share that wave, so the tail lasts half a
// tile instead of a whole one (the pages' persistent scheduler, TIRx notes
// V6, leaves the last wave partly idle: 1024 tiles over 148 CTAs is 6.9
// tiles each).
struct WorkItem {
    int32_t m_idx;
    int32_t n_idx;
    int32_t n_off;    // 0, or bn / 2 for the second half of a split tile
    int32_t n_len;    // the tile width bn, or bn / 2 for a half tile
    int32_t slice;    // K slice of a split-K tile (0 without split-K)
    int32_t kt_begin; // first and one-past-last 64-wide K tile of the item
    int32_t kt_end;
};

// Items [0, split_from) are whole tiles t = item in grouped order; items from
// split_from on are the two halves of tiles split_from, split_from + 1, ...
// With slices > 1 (split-K; nothing is then split along N) item t*slices + s
// is K slice s of tile t: K tiles [s*k_tiles/slices, (s+1)*k_tiles/slices).
// Tiles are bn columns wide (256, or 64 for the narrow and tiny tiles of
// small problems).
GEMM_HD WorkItem work_of(int32_t item, int32_t num_m, int32_t num_n, int32_t group, int32_t split_from,
                         int32_t k_tiles = 0, int32_t slices = 1, int32_t bn = 256) {
    if (slices > 1) {
        const int32_t t = item / slices;
        const int32_t sl = item - t * slices;
        const TileCoord c = tile_of(t, num_m, num_n, group);
        WorkItem w;
        w.m_idx = c.m_idx;
        w.n_idx = c.n_idx;
        w.n_off = 0;
        w.n_len = bn;
        w.slice = sl;
        w.kt_begin = static_cast<int32_t>(static_cast<int64_t>(sl) * k_tiles / slices);
        w.kt_end = static_cast<int32_t>(static_cast<int64_t>(sl + 1) * k_tiles / slices);
        return w;
    }
    int32_t t = item;
    int32_t half = -1;
    if (item >= split_from) {
        const int32_t r = item - split_from;
        t = split_from + r / 2;
        half = r % 2;
    }
    const TileCoord c = tile_of(t, num_m, num_n, group);
    WorkItem w;
    w.m_idx = c.m_idx;
    w.n_idx = c.n_idx;
    w.n_off = half < 0 ? 0 : (bn / 2) * half;
    w.n_len = half < 0 ? bn : bn / 2;
    w.slice = 0;
    w.kt_begin = 0;
    w.kt_end = k_tiles;
    return w;
}

// Split-K (TIRx notes V6 leaves a partly idle last wave; with very few tiles
// most of the GPU would idle for the whole K-loop).  With num_tiles tiles on
// `clusters` persistent clusters and k_tiles K tiles per tile, K is cut into
// S = min(clusters / num_tiles, k_tiles / 8, 16) slices when that gives at
// least 4 (a 2-way N split already halves the K-loop's time, so fewer slices
// would not gain); otherwise 1.  Each slice then runs at least 8 K tiles.
GEMM_HD int32_t splitk_slices(int32_t num_tiles, int32_t clusters, int32_t k_tiles) {
    if (num_tiles <= 0 || clusters <= 0) return 1;
    int32_t s = clusters / num_tiles;
    if (s > k_tiles / 8) s = k_tiles / 8;
    if (s > 16) s = 16;
    return s >= 4 ? s : 1;
}

// Tiles [split_from, num_tiles) are split in two when that fits the last
// wave: with num_tiles = q * clusters + r and 0 < 2r <= clusters, the r tiles
// of the last wave become 2r half tiles, one per cluster.  Returns split_from
// (num_tiles when nothing is split); the item count is then
// num_tiles + (num_tiles - split_from).
GEMM_HD int32_t split_point(int32_t num_tiles, int32_t clusters) {
    const int32_t r = num_tiles % clusters;
    if (r == 0 || 2 * r > clusters) return num_tiles;
    return num_tiles - r;
}

// Where one CTA of a work item reads and writes (TIRx notes V8, "Operand
// Partition", "Output Ownership", "Epilogue Column Address").  An item covers
// (bm * cg * nc) rows x n_len columns of D, nc being the number of MMA
// consumers (TIRx notes V9: two consumers stack their bm*cg rows along M),
// in a grid of tiles bn columns wide; bm is 128, or 64 for the tiny tiles.
// CTA `rank` loads, for consumer c, A rows a_row + c*bm*cg .. +bm and the
// shared B rows b_row .. +n_len/cg, and writes D rows d_row + c*bm*cg .. +bm
// over all n_len columns from d_col: the rank selects the A rows and the
// output rows, and only the slice of B it loads, never the output columns.
struct CtaOrigin {
    int32_t a_row;
    int32_t b_row;
    int32_t d_row;
    int32_t d_col;
};

GEMM_HD CtaOrigin cta_origin(WorkItem w, int32_t cg, int32_t rank, int32_t nc = 1, int32_t bn = 256,
                             int32_t bm = 128) {
    CtaOrigin o;
    const int32_t m_base = w.m_idx * bm * cg * nc;
    const int32_t n_base = w.n_idx * bn + w.n_off;
    o.a_row = m_base + rank * bm;
    o.b_row = n_base + rank * (w.n_len / cg);
    o.d_row = o.a_row;
    o.d_col = n_base;
    return o;
}

}  // namespace gemm_f16
