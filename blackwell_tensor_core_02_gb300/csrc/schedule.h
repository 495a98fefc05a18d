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
// notes V6, "Better L2 Locality", l2_group_size = 8).  A bijection from
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
    c.n_idx = r / gsize;
    return c;
}

// Where one CTA of a tile reads and writes (TIRx notes V8, "Operand
// Partition", "Output Ownership", "Epilogue Column Address").  A tile is
// (128 * cg) rows x 256 columns of D.  CTA `rank` of the pair loads A rows
// a_row .. +128 and B rows b_row .. +256/cg, and writes D rows d_row .. +128
// over all 256 columns from d_col: the rank selects the A rows and the output
// rows, and only the slice of B it loads, never the output columns.
struct CtaOrigin {
    int32_t a_row;
    int32_t b_row;
    int32_t d_row;
    int32_t d_col;
};

GEMM_HD CtaOrigin cta_origin(TileCoord tc, int32_t cg, int32_t rank) {
    CtaOrigin o;
    const int32_t m_base = tc.m_idx * 128 * cg;
    const int32_t n_base = tc.n_idx * 256;
    o.a_row = m_base + rank * 128;
    o.b_row = n_base + rank * (256 / cg);
    o.d_row = o.a_row;
    o.d_col = n_base;
    return o;
}

}  // namespace gemm_f16
