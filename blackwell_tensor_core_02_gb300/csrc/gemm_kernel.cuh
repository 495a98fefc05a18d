// gemm_kernel.cuh -- the persistent, warp-specialized sm_103a GEMM kernel.
//
// D (M x N, fp16) = A (M x K, fp16) * B (N x K, fp16)^T, fp32 accumulation in
// tensor memory, one round to fp16 at writeback.
//
// The data path is the pages' fixed hop chain ("GEMM I -- the tiled
// baseline", "The one invariant"): GMEM -TMA-> swizzled SMEM -tcgen05.mma->
// TMEM (fp32) -tcgen05.ld-> registers -cast-> SMEM -TMA-> GMEM.
//
// Roles (one CTA = 6 warps, "GEMM III", Step 7; TIRx notes V7 "Warp Roles"):
//   warp 0     TMA producer: one elected lane fills the SMEM ring.
//   warp 1     TMEM allocator; in the leader CTA also the MMA issuer (one
//              elected lane issues every tcgen05.mma, "GEMM I", "Why one
//              elected thread issues the MMA").
//   warps 2-5  epilogue: each warp owns one 32-lane quarter of TMEM (warp w
//              may only touch lanes 32*(w%4) .. +31), i.e. 32 rows of the tile
//              (16 with 64-row tiles).
//
// Two producer-consumer rings ("GEMM III", "Four barriers"; TIRx notes V7):
//   SMEM ring:  empty[s] (mma2tma) -> TMA -> full[s] (tma2mma) -> MMA -> empty[s]
//   TMEM ring:  tmem_empty[a] (ld2mma) -> MMA -> tmem_full[a] (mma2ld) -> epilogue
// The TMEM ring has two accumulator buffers, so the epilogue of tile i runs
// while the MMA issuer already accumulates tile i+1 into the other buffer.
// The epilogue reads its whole share of the accumulator and rounds it to
// packed fp16 in registers before it stages and stores anything, so the
// buffer goes back to the MMA after the TMEM reads alone; the slower SMEM
// staging and TMA stores then run beside the next tile's MMAs.
//
// CTA pair (CG = 2; "GEMM III", Step 8; TIRx notes V8): a 2-CTA cluster owns a
// 256 x 256 tile.  CTA r loads A rows m_base + 128r and B rows n_base + 128r
// into its own SMEM; the leader (rank 0) alone issues cta_group::2 MMAs of
// M = 256, N = 256 that read both CTAs' SMEM and write each CTA's own TMEM
// ([A_r B_0^T | A_r B_1^T]).  Both CTAs' TMA bytes complete on the leader's
// full[s]; the MMA commits arrive on empty[s] / tmem_full[a] of both CTAs
// (cta_mask 0b11); tmem_empty[a] on the leader counts the epilogue warps of
// both CTAs.
//
// Two MMA consumers (NC = 2, CG = 2; "GEMM III", Step 9; TIRx notes V9): the
// cluster tile grows to 512 x 256.  Each stage holds two A blocks (one per
// consumer, 256 rows apart) and one B block that both consumers read, so B
// is loaded once for twice the math.  Consumer c accumulates into TMEM
// columns [256c, 256c + 256); with all 512 columns taken there is no second
// accumulator buffer, so the next tile waits for the epilogue to drain TMEM.
// The CTA has three warpgroups: warps 0-1 as above (2-3 idle), warps 4-7
// drain consumer 0 and warps 8-11 consumer 1.  Registers move between them
// ("GEMM III", Step 7, setmaxnreg): 384 threads launch with 168 registers
// each; the producer/MMA warpgroup drops to 40 and the two epilogue
// warpgroups rise to 232, enough to hold a warp's whole 32 x 256 slice as
// packed fp16.  So, as in the default kernel, the epilogue reads and rounds
// its slice, hands TMEM back (the next tile's MMAs start) and only then
// stages and stores it by TMA, through one 4 KiB buffer per warp beside the
// four 48 KiB stages.
//
// Narrow tiles (BN = 64, CG = 1, NC = 1): for problems whose 128 x 64 tiles fit
// one wave of CTAs.  Same roles; an 8-stage ring of 24 KiB stages holds a K of
// 512 at once, TMEM is 128 columns (two 64-column accumulators), and the
// epilogue stages each warp's rows in shared memory and writes D with
// coalesced warp stores.  Not on the pages, which fix the tile.
//
// Tiny tiles (BM = 64, BN = 64): for problems whose 64 x 64 tiles fill at most
// two thirds of a wave, the same again with MMAs of M = 64 and a ring of 6
// stages of two 16 KiB K tiles.  An M = 64 accumulator takes lanes 0-15 of each 32-lane
// quarter of TMEM (row r in lane 32 * (r / 16) + r % 16), so each epilogue
// warp reads its quarter as usual and stores 16 rows from its lanes 0-15.
//
// Thin tiles (BM = 64, BN = 16): the tiny tiles cut four times finer along N
// for the shortest problems, MMAs of M = 64, N = 16, two 16-column
// accumulators in the smallest TMEM allocation (32 columns), a ring of 3 stages
// of four 10 KiB K tiles, and an epilogue that stores each row's 32 bytes
// straight from registers.  Each CTA then
// loads and drains a quarter as much per tile, which shortens the one pass
// of the data path such a problem is.
//
// K split across a cluster (KS = 2, 4, 8; narrow and tiny tiles): KS CTAs own
// one tile, CTA s runs K slice s, and the copy engine moves each CTA's fp32
// sums to the CTA that owns those rows, which adds the KS slices in order,
// rounds once and stores D (see the end of the kernel).
//
// Split-K (NC = 1): with very few tiles, item t*S + s runs K slice s of tile
// t and its epilogue writes the fp32 partial sum of that slice to a workspace
// [S][M][N]; splitk_reduce_kernel then adds the S partials in fp32 and rounds
// once to fp16 (the sum is still accumulated in fp32 and rounded once).
//
// Every wait is bounded: after `timeout_ns` the waiting role records an error
// in the device status word, raises the CTA's abort flag and falls through to
// teardown, so a protocol error ends the kernel instead of hanging the GPU.
#pragma once

#include <stdint.h>

#include "ptx.cuh"
#include "schedule.h"

namespace gemm_f16 {

__device__ int g_status;              // first error code of any CTA (0 = none)
__device__ unsigned long long g_info; // where it happened (role, CTA, tile seq)

enum : int { kStatusTimeout = -7, kStatusBounds = -10 };
enum : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3 };

// The checked build (-DGEMM_F16_DEVICE_CHECKS=1, a second library the tests
// load beside the production one) tests, before each access, that the work
// item, ring stage, TMEM columns, epilogue chunk and staging buffer are in
// range.  A failed check records kStatusBounds with (role, check, CTA, tile
// sequence) in the status word and raises the CTA's abort flag, so the CTA
// ends through the same path as a timed-out wait; it never traps.  In the
// production build every check compiles to nothing.
#ifndef GEMM_F16_DEVICE_CHECKS
#define GEMM_F16_DEVICE_CHECKS 0
#endif
enum : uint32_t {
    kCheckItem = 1,
    kCheckStage = 2,
    kCheckTmem = 3,
    kCheckChunk = 4,
    kCheckStaging = 5,
    kCheckReduceRow = 6
};

// BN is the tile width: 256, or 64 for the narrow single-CTA tiles of small
// problems (more CTAs, and a ring deep enough to hold a K of 512 at once).
// BM is the rows of D per CTA and consumer: 128, or 64 for the tiny tiles
// (64 x 64) of the smallest problems.  KS > 1 (narrow and tiny tiles) splits
// K across a cluster of KS CTAs that add their partial sums through
// distributed shared memory.
template <int CG, int NC, int BN = 256, int BM = 128, int KS = 1>
struct Cfg {
    static_assert(CG == 1 || CG == 2, "cta_group is 1 or 2");
    static_assert(NC == 1 || (NC == 2 && CG == 2), "two consumers need a CTA pair");
    static_assert(BN == 256 || ((BN == 64 || BN == 16) && CG == 1 && NC == 1), "narrow tiles are single-CTA, one consumer");
    static_assert(BM == 128 || (BM == 64 && BN <= 64), "64-row tiles are narrow");
    static_assert(BN != 16 || (BM == 64 && KS == 1), "thin tiles are 64 x 16, without a K split");
    static_assert(KS == 1 || ((KS == 2 || KS == 4 || KS == 8) && BN == 64), "a K split over 2, 4 or 8 narrow or tiny CTAs");
    static constexpr bool NARROW = BN != 256;
    static constexpr bool TINY = BM == 64;
    static constexpr bool THIN = BN == 16;
    static constexpr bool KSPLIT = KS > 1;
    static constexpr int CLUSTER = CG * KS;             // CTAs per cluster
    // co-resident cluster count slot of this configuration in the host's
    // per-device table (thin tiles share the tiny tiles' slot: they need less
    // shared memory, and the host checks that at least as many fit)
    static constexpr int KIND = KSPLIT ? (KS == 2 ? 5 : (KS == 4 ? 6 : 7)) + (TINY ? 0 : 3)
                                       : (TINY ? 4 : (NARROW ? 3 : (CG == 1 ? 0 : NC)));
    static constexpr int BLOCK_M = BM;                  // rows of D per CTA and consumer
    static constexpr int BLOCK_N = BN;                  // columns of D per tile (MMA N)
    static constexpr int BLOCK_K = 64;                  // one 128-byte swizzle row of fp16
    static constexpr int MMA_M = BLOCK_M * CG;          // M of one tcgen05.mma (one consumer)
    static constexpr int TILE_M = MMA_M * NC;           // rows of D per tile
    static constexpr int UMMA_K = 16;                   // K of one tcgen05.mma kind::f16
    static constexpr int B_ROWS = BLOCK_N / CG;         // rows of B each CTA loads
    // K tiles of 64 per ring stage.  The MMAs of one K tile of a 64-row tile (tiny or thin) are
    // so short that the per-stage hand-off (full wait, fence, commit to empty, the producer's
    // turn) bounds the K-loop, so tiny tiles move two K tiles per stage and thin ones four
    // (fewer, larger stages; the last stage of a work item may hold fewer).  Measured on GB300
    // (graph-timed, us, one vs two K tiles per stage): 256x256x512 (thin) 2.70 vs 2.43,
    // 512x256x256 2.60 vs 2.46, 256x256x4096 (tiny, K over 4 CTAs) 4.81 vs 4.19, 128x128x64
    // (one K tile) 1.58 either way; thin tiles, two vs four: 256x256x512 2.43 vs 2.40,
    // 256x256x768 2.80 vs 2.72, 128x256x768 2.77 vs 2.69 (three: 2.44, 2.76, 2.74); tiny tiles
    // lose with four (256x256x4096 4.21 vs 4.45); CTA pairs lose with 3 stages of 2 (4096^3
    // +13 %, 1536^3 +6 %), and narrow tiles 1-3 %.
    static constexpr int KPS = THIN ? 4 : (TINY ? 2 : 1);
    static constexpr int A_BLOCK = BLOCK_M * BLOCK_K * 2;
    static constexpr int A_KT = A_BLOCK * NC;           // one K tile of A (every consumer's block)
    static constexpr int A_STAGE = A_KT * KPS;
    static constexpr int B_KT = B_ROWS * BLOCK_K * 2;   // one K tile of B
    static constexpr int B_STAGE = B_KT * KPS;
    static constexpr int STAGES = (TINY ? 12 : (NARROW ? 8 : (NC == 2 ? 4 : (CG == 2 ? 6 : 4)))) / KPS;
    static constexpr uint32_t TX_BYTES = (A_KT + B_KT) * CG;      // per K tile, on the leader
    static constexpr uint32_t TX_HALF = (A_KT + B_KT / 2) * CG;   // the same for a half tile
    static constexpr int ACC_BUFS = NC == 2 ? 1 : 2;
    static constexpr int TMEM_COLS = ACC_BUFS * NC * BLOCK_N;           // 512 (all of TMEM), 128 or 32
    static_assert(TMEM_COLS == 512 || TMEM_COLS == 128 || TMEM_COLS == 32, "a power of two of at least 32 columns");
    static constexpr int EPI_WARPS = 4 * NC;
    static constexpr int EPI_WARP0 = NC == 2 ? 4 : 2;   // first epilogue warp (a warpgroup boundary for NC 2)
    static constexpr bool EPI_TMA = !NARROW;            // stage in SMEM, store D (or split-K partials) by TMA
    // Narrow and tiny tiles stage each warp's rows in SMEM and read them back
    // so that a warp's store covers whole 128-byte rows of D (coalesced
    // st.global): a row per lane would send 16-byte pieces of 16 or 32
    // different rows per store instruction.
    static constexpr bool EPI_COALESCED = NARROW && !THIN;
    static constexpr int EPI_N = THIN ? 16 : 64;        // columns per epilogue chunk
    static constexpr int WARP_ROWS = BLOCK_M / 4;       // rows of D per epilogue warp: the first WARP_ROWS
                                                        // lanes of its TMEM quarter
    // staging buffers per epilogue warp: two (one chunk's TMA store reads one while the next
    // chunk fills the other), or one with two consumers, whose operand ring leaves room for
    // no more
    static constexpr int EPI_BUFS = EPI_TMA ? (NC == 2 ? 1 : 2) : (EPI_COALESCED ? 1 : 0);
    static constexpr int EPI_BUF = 32 * 64 * 2;         // one warp's 32 rows x 64 fp16 = 4 KiB
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    // Register split of the two-consumer kernel (setmaxnreg).  A CTA's pool is what it
    // launches with: THREADS x the registers per thread the compiler assigns, at most
    // REGS_AT_LAUNCH under __launch_bounds__(THREADS, 1).  The host refuses to launch this
    // kernel unless the compiled count is exactly REGS_AT_LAUNCH, so the split below always
    // fits the pool and no setmaxnreg.inc can wait for registers that never come.
    static constexpr bool REG_SPLIT = NC == 2;
    static constexpr int REGS_AT_LAUNCH = (65536 / THREADS) / 8 * 8;  // 168 for 384 threads
    static constexpr int REGS_PRODUCER = 40;            // warps 0-3 after the split
    static constexpr int REGS_EPILOGUE = 232;           // each epilogue warp after the split
    static_assert(!REG_SPLIT || (EPI_WARP0 == 4 && 32 * EPI_WARP0 * REGS_PRODUCER +
                                                      32 * EPI_WARPS * REGS_EPILOGUE <=
                                                  THREADS * REGS_AT_LAUNCH),
                  "the register split must fit the CTA's pool at launch");
    // Shared-memory layout (offsets from a 1024-byte aligned base; identical
    // in both CTAs of a pair, which the pair MMA relies on).
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_D = OFF_B + STAGES * B_STAGE;
    // With a K split the epilogue region at OFF_D receives the cluster's fp32
    // partial sums of this CTA's rows (KS slices x BLOCK_M / KS rows x BLOCK_N),
    // in place of the staging buffers.  The CTA's own sums (all BLOCK_M rows,
    // staged for the copies to their owners) go to OFF_SRC, the start of the
    // operand ring: a CTA of a K split has one work item, so when its
    // accumulator is complete every load has landed and every MMA has read
    // its operands, and the ring is idle for good.
    static constexpr int EPI_REGION = KSPLIT ? BLOCK_M * BLOCK_N * 4 : EPI_WARPS * EPI_BUFS * EPI_BUF;
    static constexpr int OFF_SRC = OFF_A;
    static constexpr int OFF_BAR = OFF_D + EPI_REGION;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1 + (KSPLIT ? 1 : 0);  // + drain (+ recv)
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;         // tmem base, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = SMEM_BYTES + 1024;            // alignment slack
    static_assert(SMEM_ALLOC <= 232448, "exceeds the 227 KiB per-block shared memory limit");
    static_assert(A_BLOCK % 1024 == 0 && B_STAGE % 1024 == 0 && EPI_BUF % 1024 == 0, "1 KiB swizzle atoms");
    // with a K split, the staging buffers receive the cluster's fp32 partial
    // sums of this CTA's rows: KS slices x (BLOCK_M / KS) rows x BLOCK_N fp32
    static constexpr int KS_ROWS = BLOCK_M / KS;        // rows of the tile this CTA adds up and stores
    static constexpr uint32_t KS_ROW_BYTES = BLOCK_N * 4;             // one row of fp32 sums
    static constexpr uint32_t KS_RECV_BYTES = BLOCK_M * KS_ROW_BYTES;  // all slices of those rows
    static_assert(!KSPLIT || (EPI_COALESCED && KS_ROWS % 8 == 0),
                  "the cluster's partial sums of a CTA's rows fit its staging buffers");
    static_assert(!KSPLIT || BLOCK_M * KS_ROW_BYTES <= STAGES * (A_STAGE + B_STAGE),
                  "a K split's own sums fit the idle operand ring");
};

struct Params {
    int32_t M, N, K;
    int32_t num_m_tiles, num_n_tiles, k_tiles, num_tiles;
    int32_t num_items, split_from;  // work items; items from split_from on are half tiles
    int32_t slices;                 // split-K slices (1: none)
    int32_t raster_group;
    uint32_t debug_flags;
    uint64_t timeout_ns;
    uint16_t *D;       // for the epilogues that store with st.global (row-major, ldd = N)
    float *partial;    // split-K workspace [slices][M][N] fp32, when slices > 1
};

enum : uint32_t { kDebugProducerPhase0 = 1u };

// Instruction descriptor of tcgen05.mma kind::f16 (PTX ISA): D fp32 [4,6)=1,
// A and B fp16 [7,10)=[10,13)=0, both K-major [15]=[16]=0, N>>3 at [17,23),
// M>>4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void record_failure(uint32_t role, uint32_t seq) {
    if (atomicCAS(&g_status, 0, kStatusTimeout) == 0) {
        g_info = (static_cast<unsigned long long>(role) << 56) |
                 (static_cast<unsigned long long>(blockIdx.x & 0xFFFFFFu) << 32) | seq;
    }
}

__device__ __forceinline__ bool in_bounds(bool ok, volatile int *abort_flag, uint32_t role, uint32_t check,
                                          uint32_t seq) {
#if GEMM_F16_DEVICE_CHECKS
    if (!ok) {
        if (atomicCAS(&g_status, 0, kStatusBounds) == 0) {
            g_info = (static_cast<unsigned long long>(role) << 56) | (static_cast<unsigned long long>(check) << 48) |
                     (static_cast<unsigned long long>(blockIdx.x & 0xFFFFu) << 32) | seq;
        }
        *abort_flag = 1;
        return false;
    }
#else
    (void)abort_flag, (void)role, (void)check, (void)seq;
#endif
    return ok || !GEMM_F16_DEVICE_CHECKS;
}

// A work item the scheduler hands out: a tile inside the grid, a K range
// inside K, columns inside the tile.
__device__ __forceinline__ bool item_ok(const WorkItem &w, int32_t num_m, int32_t num_n, int32_t k_tiles, int32_t bn) {
    return w.m_idx >= 0 && w.m_idx < num_m && w.n_idx >= 0 && w.n_idx < num_n && w.kt_begin >= 0 &&
           w.kt_begin < w.kt_end && w.kt_end <= k_tiles && w.n_off >= 0 && w.n_len > 0 && w.n_off + w.n_len <= bn;
}

// Bounded wait by one thread.  Returns false if the wait ran out (the failure
// is recorded and the CTA's abort flag raised) or, when `honor_abort`, as soon
// as another role of this CTA has aborted.  kCluster: acquire at cluster scope
// (the arrivals come from other CTAs of the cluster).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             uint64_t timeout_ns, uint32_t role, uint32_t seq,
                                             bool honor_abort = true) {
    auto try_wait = [](uint32_t b, uint32_t ph) {
        return kCluster ? ptx::mbar_try_wait_cluster(b, ph) : ptx::mbar_try_wait(b, ph);
    };
    if (try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (try_wait(bar, parity)) return true;
        if ((i & 15u) == 0) {
            if (honor_abort && *abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                record_failure(role, seq);
                return false;
            }
        }
    }
}

// fp32 -> fp16 with round to nearest even, two values packed per word:
// out[j] = (fp16(in[2j+1]) << 16) | fp16(in[2j]), j < 16.
__device__ __forceinline__ void to_f16x2(const uint32_t (&in)[32], uint32_t *out) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const __half2 v = __floats2half2_rn(__uint_as_float(in[2 * j]), __uint_as_float(in[2 * j + 1]));
        out[j] = *reinterpret_cast<const uint32_t *>(&v);
    }
}

template <int CG, int NC, int BN, int BM, int KS = 1>
__global__ void __launch_bounds__(Cfg<CG, NC, BN, BM, KS>::THREADS, 1)
    gemm_f16_nt_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmD,
                       const __grid_constant__ CUtensorMap tmP, const Params p) {
    using C = Cfg<CG, NC, BN, BM, KS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) % 32;
    const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int cluster = static_cast<int>(blockIdx.x) / CG;
    const int num_clusters = static_cast<int>(gridDim.x) / CG;

    const uint32_t sA = base + C::OFF_A;
    const uint32_t sB = base + C::OFF_B;
    const uint32_t sD = base + C::OFF_D;
    const uint32_t bar_full = base + C::OFF_BAR;              // [STAGES]
    const uint32_t bar_empty = bar_full + 8 * C::STAGES;      // [STAGES]
    const uint32_t bar_tfull = bar_empty + 8 * C::STAGES;     // [ACC_BUFS]
    const uint32_t bar_tempty = bar_tfull + 8 * C::ACC_BUFS;  // [ACC_BUFS]
    const uint32_t bar_drain = bar_tempty + 8 * C::ACC_BUFS;
    const uint32_t bar_recv = bar_drain + 8;  // K split: the cluster's partial rows have arrived
    const uint32_t krank = C::KSPLIT ? ptx::cluster_ctarank() : 0u;  // K slice of this CTA
    // A CTA pair splits its teardown cluster barrier: the epilogue warps arrive
    // as soon as their last TMEM read is done, so the barrier's latency passes
    // under the last tile's stores; every thread arrives exactly once.
    bool cluster_arrived = false;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    // ---- prologue: barriers, TMEM, tensor-map prefetch (once per persistent CTA)
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmBh);
        ptx::prefetch_tensormap(&tmD);
        if (p.slices > 1) ptx::prefetch_tensormap(&tmP);
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, 1);
        }
        for (int a = 0; a < C::ACC_BUFS; ++a) {
            ptx::mbar_init(bar_tfull + 8 * a, 1);
            ptx::mbar_init(bar_tempty + 8 * a, C::EPI_WARPS * CG);
        }
        ptx::mbar_init(bar_drain, 1);
        if constexpr (C::KSPLIT) {
            // the cluster's copies of this CTA's rows complete KS_RECV_BYTES
            // of transactions on it; its one arrival is made here
            ptx::mbar_init(bar_recv, 1);
            ptx::mbar_arrive_expect_tx(bar_recv, C::KS_RECV_BYTES);
        }
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tcgen05_fence_before();
    if constexpr (C::CLUSTER > 1) {
        ptx::cluster_sync();  // also: every barrier of the cluster initialised before any remote arrival
    } else {
        __syncthreads();
    }
    ptx::tcgen05_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    // Everything above touches only this CTA's own resources, so with a
    // programmatic launch it overlaps the tail of the previous kernel of the
    // stream; so does what each role does below before its own
    // griddepcontrol.wait (the producer's before its first TMA load, the
    // epilogue's before its first write of D; the MMA issuer touches no
    // global memory).  A, B and D are read and written only after it.
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();

    if (warp < C::EPI_WARP0) {
        // Warpgroup 0 with two consumers: its producer, its MMA issuer and two idle
        // warps give registers to the two epilogue warpgroups, all four warps at once.
        // (The register limit of each role's code then follows from the instruction
        // that starts its branch.)
        if constexpr (C::REG_SPLIT) ptx::setmaxnreg_dec<C::REGS_PRODUCER>();
        if (warp == 0) {
            // ---------------------------------------------------- TMA producer
            if (ptx::elect_one()) {
                // The producer end starts one phase ahead of the consumer end
                // ("GEMM III", "The subtlest bug: opposite initial phases").  The
                // debug flag starts it at phase 0 instead, which blocks every role;
                // only the tests of the timeout path set it.
                PipelineState ring(C::STAGES, (p.debug_flags & kDebugProducerPhase0) ? 0u : 1u);
                uint32_t seq = 0;
                bool ok = true;
                bool dependency_met = false;  // griddepcontrol.wait has returned
                int item = cluster;
                WorkItem w = work_of(item, p.num_m_tiles, p.num_n_tiles, p.raster_group, p.split_from, p.k_tiles,
                                     p.slices, C::BLOCK_N);
                if (item < p.num_items) {
                    // Before the wait, only ask L2 for the A and B boxes of the
                    // first ring fill: L2 is where every later load reads them,
                    // and a line the previous kernel still writes is updated
                    // there, so the prefetch changes no value; it moves the HBM
                    // latency of the first k-tiles under the previous kernel's
                    // tail.
                    const CtaOrigin o = cta_origin(w, CG, static_cast<int32_t>(rank), NC, C::BLOCK_N, C::BLOCK_M);
                    const CUtensorMap *mapB = w.n_len < C::BLOCK_N ? &tmBh : &tmB;
                    const int kt_end = w.kt_begin + C::STAGES * C::KPS < w.kt_end ? w.kt_begin + C::STAGES * C::KPS : w.kt_end;
                    for (int kt = w.kt_begin; kt < kt_end; ++kt) {
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            ptx::tma_prefetch_l2_2d(&tmA, kt * C::BLOCK_K, o.a_row + c * C::MMA_M);
                        }
                        ptx::tma_prefetch_l2_2d(mapB, kt * C::BLOCK_K, o.b_row);
                    }
                }
                for (; ok && item < p.num_items; item += num_clusters, ++seq) {
                    if (seq > 0) {
                        w = work_of(item, p.num_m_tiles, p.num_n_tiles, p.raster_group, p.split_from, p.k_tiles,
                                    p.slices, C::BLOCK_N);
                    }
                    if (!in_bounds(item_ok(w, p.num_m_tiles, p.num_n_tiles, p.k_tiles, C::BLOCK_N), abort_flag,
                                   kRoleProducer, kCheckItem, seq)) {
                        ok = false;
                        break;
                    }
                    const CtaOrigin o = cta_origin(w, CG, static_cast<int32_t>(rank), NC, C::BLOCK_N, C::BLOCK_M);
                    const bool half = w.n_len < C::BLOCK_N;
                    const CUtensorMap *mapB = half ? &tmBh : &tmB;
                    for (int kt = w.kt_begin; kt < w.kt_end; kt += C::KPS) {
                        const int nkt = w.kt_end - kt < C::KPS ? w.kt_end - kt : C::KPS;  // K tiles in this stage
                        if (!in_bounds(ring.stage >= 0 && ring.stage < C::STAGES, abort_flag, kRoleProducer, kCheckStage,
                                       seq) ||
                            !wait_bounded(bar_empty + 8 * ring.stage, ring.phase, abort_flag, p.timeout_ns,
                                          kRoleProducer, seq)) {
                            ok = false;
                            break;
                        }
                        const uint32_t full = bar_full + 8 * ring.stage;
                        if (leader) ptx::mbar_arrive_expect_tx(full, (half ? C::TX_HALF : C::TX_BYTES) * nkt);
                        if (!dependency_met) {
                            // the first load of A or B: the previous kernel of
                            // the stream must be complete and its writes visible
                            ptx::griddep_wait();
                            dependency_met = true;
                        }
#pragma unroll
                        for (int j = 0; j < C::KPS; ++j) {
                            if (j >= nkt) break;
                            const int32_t k0 = (kt + j) * C::BLOCK_K;
                            const uint32_t sa = sA + ring.stage * C::A_STAGE + j * C::A_KT;
                            const uint32_t sb = sB + ring.stage * C::B_STAGE + j * C::B_KT;
                            if constexpr (CG == 2) {
                                const uint32_t full_leader = ptx::mapa(full, 0);
#pragma unroll
                                for (int c = 0; c < NC; ++c) {  // consumer c's A rows lie c * MMA_M below
                                    ptx::tma_load_2d_pair(sa + c * C::A_BLOCK, &tmA, full_leader, k0,
                                                          o.a_row + c * C::MMA_M);
                                }
                                ptx::tma_load_2d_pair(sb, mapB, full_leader, k0, o.b_row);
                            } else {
                                ptx::tma_load_2d(sa, &tmA, full, k0, o.a_row);
                                ptx::tma_load_2d(sb, mapB, full, k0, o.b_row);
                            }
                        }
                        ring.advance();
                    }
                }
                if (!ok) {
                    // Give loads already in flight time to land before teardown.
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (ptx::globaltimer_ns() - t0 < 20000) ptx::nanosleep(1000);
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ------------------------------------------------------ MMA issuer
            if (leader && ptx::elect_one()) {
                constexpr uint32_t idesc_full = idesc_f16_f32(C::MMA_M, C::BLOCK_N);
                constexpr uint32_t idesc_half = idesc_f16_f32(C::MMA_M, C::BLOCK_N / 2);
                constexpr uint16_t pair_mask = CG == 2 ? 0x3 : 0x1;
                PipelineState ring(C::STAGES, 0u);
                PipelineState acc(C::ACC_BUFS, 1u);
                uint32_t seq = 0;
                bool ok = true;
                for (int item = cluster; ok && item < p.num_items; item += num_clusters, ++seq) {
                    const WorkItem w = work_of(item, p.num_m_tiles, p.num_n_tiles, p.raster_group, p.split_from,
                                               p.k_tiles, p.slices, C::BLOCK_N);
                    const uint32_t idesc = w.n_len < C::BLOCK_N ? idesc_half : idesc_full;
                    if (!in_bounds(item_ok(w, p.num_m_tiles, p.num_n_tiles, p.k_tiles, C::BLOCK_N), abort_flag, kRoleMma,
                                   kCheckItem, seq) ||
                        !in_bounds(acc.stage >= 0 && (acc.stage + 1) * NC * C::BLOCK_N <= C::TMEM_COLS, abort_flag,
                                   kRoleMma, kCheckTmem, seq) ||
                        !wait_bounded(bar_tempty + 8 * acc.stage, acc.phase, abort_flag, p.timeout_ns, kRoleMma,
                                      seq)) {
                        ok = false;
                        break;
                    }
                    ptx::tcgen05_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc.stage * NC * C::BLOCK_N);
                    for (int kt = w.kt_begin; kt < w.kt_end; kt += C::KPS) {
                        const int nkt = w.kt_end - kt < C::KPS ? w.kt_end - kt : C::KPS;  // K tiles in this stage
                        if (!in_bounds(ring.stage >= 0 && ring.stage < C::STAGES, abort_flag, kRoleMma, kCheckStage, seq) ||
                            !wait_bounded(bar_full + 8 * ring.stage, ring.phase, abort_flag, p.timeout_ns, kRoleMma,
                                          seq)) {
                            ok = false;
                            break;
                        }
                        ptx::tcgen05_fence_after();
#pragma unroll
                        for (int j = 0; j < C::KPS; ++j) {
                            if (j >= nkt) break;
                            const uint64_t b_desc = ptx::smem_desc_k_sw128(sB + ring.stage * C::B_STAGE + j * C::B_KT);
#pragma unroll
                            for (int c = 0; c < NC; ++c) {  // both consumers read the same B stage
                                const uint64_t a_desc = ptx::smem_desc_k_sw128(sA + ring.stage * C::A_STAGE +
                                                                               j * C::A_KT + c * C::A_BLOCK);
#pragma unroll
                                for (int k = 0; k < C::BLOCK_K / C::UMMA_K; ++k) {
                                    // +32 bytes along K inside the 128-byte swizzle row: +2 in units of 16 B.
                                    const uint64_t koff = static_cast<uint64_t>(k * C::UMMA_K * 2 / 16);
                                    ptx::mma_f16<CG>(d_tmem + c * C::BLOCK_N, a_desc + koff, b_desc + koff, idesc,
                                                     (kt + j != w.kt_begin || k != 0) ? 1u : 0u);
                                }
                            }
                        }
                        ptx::mma_commit<CG>(bar_empty + 8 * ring.stage, pair_mask);  // stage free, both CTAs
                        ring.advance();
                    }
                    if (!ok) break;
                    ptx::mma_commit<CG>(bar_tfull + 8 * acc.stage, pair_mask);  // accumulator ready, both CTAs
                    acc.advance();
                }
                // Wait for every MMA issued so far before TMEM can be released,
                // also after an abort (then only the time limit ends the wait).
                ptx::mma_commit<CG>(bar_drain, 0x1);
                wait_bounded(bar_drain, 0, abort_flag, p.timeout_ns, kRoleMma, 0xFFFFFFFFu, false);
            }
            __syncwarp();
        }
    } else {
        if constexpr (C::REG_SPLIT) ptx::setmaxnreg_inc<C::REGS_EPILOGUE>();
        // -------------------------------------------------------- epilogue
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 hold the rows of this warp
        const int consumer = (warp - C::EPI_WARP0) / 4;
        // this warp's own staging buffers
        const uint32_t stage_base = sD + static_cast<uint32_t>((warp - C::EPI_WARP0) * C::EPI_BUFS * C::EPI_BUF);
        PipelineState acc(C::ACC_BUFS, 0u);
        uint32_t buf = 0;
        uint32_t seq = 0;
        for (int item = cluster; item < p.num_items; item += num_clusters, ++seq) {
            const WorkItem w = work_of(item, p.num_m_tiles, p.num_n_tiles, p.raster_group, p.split_from,
                                       p.k_tiles, p.slices, C::BLOCK_N);
            const CtaOrigin o = cta_origin(w, CG, static_cast<int32_t>(rank), NC, C::BLOCK_N, C::BLOCK_M);
            const int chunks = w.n_len / C::EPI_N;
            const int32_t row0 = o.d_row + consumer * C::MMA_M + quarter * C::WARP_ROWS;
            const int32_t col0 = o.d_col;
            bool ok = true;
            if (lane == 0) {
                ok = wait_bounded(bar_tfull + 8 * acc.stage, acc.phase, abort_flag, p.timeout_ns, kRoleEpilogue,
                                  seq);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            if (seq == 0) {
                // before this warp's first write of D (or of the split-K
                // workspace): the previous kernel of the stream must be done
                // with it
                ptx::griddep_wait();
            }
            if (GEMM_F16_DEVICE_CHECKS) {
                bool fine = in_bounds(item_ok(w, p.num_m_tiles, p.num_n_tiles, p.k_tiles, C::BLOCK_N), abort_flag,
                                      kRoleEpilogue, kCheckItem, seq);
                fine = fine && in_bounds((acc.stage * NC + consumer) * C::BLOCK_N + w.n_len <= C::TMEM_COLS,
                                         abort_flag, kRoleEpilogue, kCheckTmem, seq);
                fine = fine && in_bounds(chunks >= 1 && chunks <= C::BLOCK_N / C::EPI_N, abort_flag, kRoleEpilogue,
                                         kCheckChunk, seq);
                fine = fine && in_bounds(!C::EPI_TMA || buf < static_cast<uint32_t>(C::EPI_BUFS), abort_flag,
                                         kRoleEpilogue, kCheckStaging, seq);
                if (!fine) break;
            }
            ptx::tcgen05_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>((acc.stage * NC + consumer) * C::BLOCK_N);
            auto release_tmem = [&]() {
                // This warp's part of the accumulator is in registers: hand
                // the TMEM buffer back (TIRx notes V7, "Writeback Flow").
                ptx::tcgen05_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (CG == 2) {
                        ptx::mbar_arrive_cluster(ptx::mapa(bar_tempty + 8 * acc.stage, 0));
                    } else {
                        ptx::mbar_arrive(bar_tempty + 8 * acc.stage);
                    }
                }
                if constexpr (C::CLUSTER > 1 && !C::KSPLIT) {
                    if (item + num_clusters >= p.num_items) {
                        // This CTA's last work item: the warp touches no TMEM
                        // and no other CTA's shared memory from here on (its
                        // release orders the arrival above on the leader's
                        // barrier), only its own staging and D.
                        __syncwarp();  // the arrival is warp-aligned
                        ptx::cluster_arrive();
                        cluster_arrived = true;
                    }
                }
            };
            if constexpr (C::EPI_TMA) {
                if (p.slices == 1) {
                    // fp16 D through TMA stores.  All chunks are read from TMEM
                    // and rounded to packed fp16 first (128 registers), so the
                    // buffer goes back to the MMA before any store is staged:
                    // the stores then overlap the next tile's MMAs instead of
                    // holding the accumulator.
                    uint32_t h[C::BLOCK_N / C::EPI_N][32];
#pragma unroll
                    for (int c = 0; c < C::BLOCK_N / C::EPI_N; ++c) {
                        if (c < chunks) {
                            uint32_t lo[32], hi[32];
                            ptx::tmem_ld_32x32b_x32(taddr + c * C::EPI_N, lo);
                            ptx::tmem_ld_32x32b_x32(taddr + c * C::EPI_N + 32, hi);
                            ptx::tmem_wait_ld();
                            to_f16x2(lo, h[c]);
                            to_f16x2(hi, h[c] + 16);
                        }
                    }
                    release_tmem();
#pragma unroll
                    for (int c = 0; c < C::BLOCK_N / C::EPI_N; ++c) {
                        if (c < chunks) {
                            // The store issued from this buffer EPI_BUFS chunks
                            // ago must have finished reading it.
                            if (lane == 0) ptx::bulk_wait_group_read<C::EPI_BUFS - 1>();
                            __syncwarp();
                            // Row `lane` of the 32 x 64 staging tile, in the
                            // 128-byte swizzle the D tensor map expects:
                            // 16-byte unit j of row r sits at unit j ^ (r % 8).
                            const uint32_t row_addr =
                                stage_base + buf * C::EPI_BUF + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t unit = static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u);
                                ptx::st_shared_v4(row_addr + unit * 16u, h[c][4 * j], h[c][4 * j + 1],
                                                  h[c][4 * j + 2], h[c][4 * j + 3]);
                            }
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int32_t col = col0 + c * C::EPI_N;
                                if (row0 < p.M && col < p.N) {
                                    ptx::tma_store_2d(&tmD, stage_base + buf * C::EPI_BUF, col, row0);
                                }
                                ptx::bulk_commit_group();
                            }
                            buf = (buf + 1u) % C::EPI_BUFS;
                        }
                    }
                    acc.advance();
                    continue;
                }
            }
            if constexpr (C::THIN) {
                // Thin tiles: one 16-column chunk.  Lane r of the warp holds row r of
                // its 16 rows (lanes 0-15 of its TMEM quarter); the 32 bytes of that
                // row go to D in two 16-byte stores straight from registers.
                uint32_t v[16];
                ptx::tmem_ld_32x32b_x16(taddr, v);
                ptx::tmem_wait_ld();
                release_tmem();
                uint32_t h[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const __half2 t = __floats2half2_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                    h[j] = *reinterpret_cast<const uint32_t *>(&t);
                }
                const int32_t row = row0 + lane;
                if (lane < C::WARP_ROWS && row < p.M) {
                    uint16_t *dst = p.D + static_cast<int64_t>(row) * p.N + col0;
                    // N % 8 == 0: a 16-byte unit is all in range or all out
                    if (col0 < p.N) ptx::st_global_v4(dst, h[0], h[1], h[2], h[3]);
                    if (col0 + 8 < p.N) ptx::st_global_v4(dst + 8, h[4], h[5], h[6], h[7]);
                }
                acc.advance();
                continue;
            }
            if constexpr (!C::THIN) {  // (thin tiles finished their item above)
#pragma unroll 1
                for (int c = 0; c < chunks; ++c) {
                    uint32_t lo[32], hi[32];
                    ptx::tmem_ld_32x32b_x32(taddr + c * C::EPI_N, lo);
                    ptx::tmem_ld_32x32b_x32(taddr + c * C::EPI_N + 32, hi);
                    ptx::tmem_wait_ld();
                    if (c == chunks - 1) release_tmem();
                    if constexpr (C::EPI_TMA) {
                        // Split-K: this slice's fp32 partial sums go to the
                        // workspace [slice][M][N] as two 32 x 32 fp32 boxes per
                        // chunk (128-byte rows, the same swizzled staging as the
                        // fp16 path; the 3-D map clips each slice at its own M).
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t *v = half ? hi : lo;
                            if (lane == 0) ptx::bulk_wait_group_read<C::EPI_BUFS - 1>();
                            __syncwarp();
                            const uint32_t row_addr = stage_base + buf * C::EPI_BUF + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t unit = static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u);
                                ptx::st_shared_v4(row_addr + unit * 16u, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                            }
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int32_t col = col0 + c * C::EPI_N + 32 * half;
                                if (row0 < p.M && col < p.N) {
                                    ptx::tma_store_3d(&tmP, stage_base + buf * C::EPI_BUF, col, row0, w.slice);
                                }
                                ptx::bulk_commit_group();
                            }
                            buf = (buf + 1u) % C::EPI_BUFS;
                        }
                    } else if constexpr (C::KSPLIT) {
                        // K split across the cluster: CTA s adds up and stores
                        // rows [s * KS_ROWS, (s + 1) * KS_ROWS) of the tile.
                        // Lane r writes its row R's fp32 sums over this CTA's K
                        // slice, chunk c at 16-byte units 16c .. 16c + 15, to row
                        // R of the CTA's source buffer (KS_ROW_BYTES, unit u at
                        // u ^ (R % 8): no bank conflicts).  After the last chunk
                        // one lane copies the warp's rows, by the copy engine, to
                        // slots krank * KS_ROWS + R % KS_ROWS of each owner's
                        // receive region (the same swizzle, as KS_ROWS is a
                        // multiple of 8), counted in bytes on its receive barrier.
                        const uint32_t src = base + C::OFF_SRC;
                        if (lane < C::WARP_ROWS) {
                            const uint32_t R = static_cast<uint32_t>(quarter * C::WARP_ROWS + lane);
                            const uint32_t row_addr = src + R * C::KS_ROW_BYTES;
                            const uint32_t sw = R & 7u;
                            const uint32_t u0 = 16u * static_cast<uint32_t>(c);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                ptx::st_shared_v4(row_addr + (((u0 + j) ^ sw) * 16u), lo[4 * j], lo[4 * j + 1],
                                                  lo[4 * j + 2], lo[4 * j + 3]);
                                ptx::st_shared_v4(row_addr + (((u0 + 8 + j) ^ sw) * 16u), hi[4 * j], hi[4 * j + 1],
                                                  hi[4 * j + 2], hi[4 * j + 3]);
                            }
                        }
                        if (c == chunks - 1) {
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                // rows [r0, r0 + WARP_ROWS) of the tile, cut at owner boundaries
                                const uint32_t r0 = static_cast<uint32_t>(quarter * C::WARP_ROWS);
                                for (uint32_t R = r0; R < r0 + C::WARP_ROWS;) {
                                    const uint32_t owner = R / C::KS_ROWS;
                                    uint32_t end = (owner + 1) * C::KS_ROWS;
                                    if (end > r0 + C::WARP_ROWS) end = r0 + C::WARP_ROWS;
                                    const uint32_t slot = krank * C::KS_ROWS + R % C::KS_ROWS;
                                    ptx::bulk_copy_to_cluster(ptx::mapa(sD + slot * C::KS_ROW_BYTES, owner),
                                                              src + R * C::KS_ROW_BYTES, (end - R) * C::KS_ROW_BYTES,
                                                              ptx::mapa(bar_recv, owner));
                                    R = end;
                                }
                            }
                        }
                    } else if constexpr (C::EPI_COALESCED) {
                        // Narrow and tiny tiles: lane r holds row r of this warp's
                        // WARP_ROWS rows.  Each row goes to the warp's staging
                        // buffer (128 bytes, 16-byte unit j at j ^ (r % 8), which
                        // keeps both passes free of bank conflicts); the warp then
                        // reads it back four rows per instruction, lane l taking
                        // unit l % 8 of row l / 8, so every st.global of the warp
                        // writes four whole 128-byte rows of D.  N % 8 == 0, so a
                        // 16-byte unit is all in range or all out.
                        uint32_t h[32];
                        to_f16x2(lo, h);
                        to_f16x2(hi, h + 16);
                        const uint32_t buf_base = stage_base;
                        if (lane < C::WARP_ROWS) {
                            const uint32_t row_addr = buf_base + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t unit = static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u);
                                ptx::st_shared_v4(row_addr + unit * 16u, h[4 * j], h[4 * j + 1], h[4 * j + 2],
                                                  h[4 * j + 3]);
                            }
                        }
                        __syncwarp();
                        const int32_t col = col0 + c * C::EPI_N + 8 * (lane & 7);
#pragma unroll
                        for (int i = 0; i < C::WARP_ROWS / 4; ++i) {
                            const int32_t r = 4 * i + (lane >> 3);
                            const uint32_t unit = static_cast<uint32_t>(lane & 7) ^ static_cast<uint32_t>(r & 7);
                            const uint4 v = ptx::ld_shared_v4(buf_base + static_cast<uint32_t>(r) * 128u + unit * 16u);
                            const int32_t row = row0 + r;
                            if (row < p.M && col < p.N) {
                                ptx::st_global_v4(p.D + static_cast<int64_t>(row) * p.N + col, v.x, v.y, v.z, v.w);
                            }
                        }
                        __syncwarp();  // the buffer is rewritten by the next chunk or work item
                    }
                }
            }
            acc.advance();
        }
        // The staging buffers must stay valid until the last stores have read
        // them; the stores' writes to D complete with the grid (and a
        // dependent launch's griddepcontrol.wait orders after them).
        if (lane == 0) ptx::bulk_wait_group_read<0>();
        __syncwarp();
    }

    if constexpr (C::KSPLIT) {
        // ---- K split: add the cluster's partial sums of this CTA's rows and
        // store them.  Every thread arrives on the cluster barrier once its
        // role is done, the epilogue's once all copies into this CTA have
        // landed, and waits on it only before exit: when it completes, every
        // copy of the cluster has landed, so no CTA leaves while a copy still
        // reads or writes its shared memory.  The adding in between reads
        // only this CTA's own shared memory.
        ptx::tcgen05_fence_before();
        if (warp < C::EPI_WARP0) ptx::cluster_arrive();
        if (warp >= C::EPI_WARP0) {
            // where this CTA's rows go, worked out while the copies are in flight
            ptx::griddep_wait();  // returns at once when this warp has waited already
            const WorkItem w = work_of(cluster, p.num_m_tiles, p.num_n_tiles, p.raster_group, p.split_from,
                                       p.k_tiles, p.slices, C::BLOCK_N);
            const CtaOrigin o = cta_origin(w, CG, 0, NC, C::BLOCK_N, C::BLOCK_M);
            // all KS slices of this CTA's rows are in: KS_RECV_BYTES of copies.
            // The arrival needs no release: it only has to follow the wait,
            // and what the barrier guards (no copy still touching a CTA's
            // shared memory at exit) is the completion this thread just saw.
            const bool ok = wait_bounded<true>(bar_recv, 0, abort_flag, p.timeout_ns, kRoleEpilogue, 0xFFFFFFFEu);
            ptx::cluster_arrive_relaxed();
            // per 8-column chunk of a row: add the KS slices in slice order
            // (fp32), round once to fp16, store 16 bytes; BLOCK_N / 8
            // consecutive threads cover one row of the tile in D
            constexpr int kChunks = C::BLOCK_N / 8;
            for (int u = static_cast<int>(threadIdx.x) - 32 * C::EPI_WARP0; ok && u < C::KS_ROWS * kChunks;
                 u += 32 * C::EPI_WARPS) {
                const int r = u / kChunks;   // row among this CTA's rows
                const int ch = u % kChunks;  // 8-column chunk
                if (!in_bounds(krank < static_cast<uint32_t>(KS) && r < C::KS_ROWS, abort_flag, kRoleEpilogue,
                               kCheckReduceRow, 0)) {
                    break;
                }
                const uint32_t sw = static_cast<uint32_t>(r) & 7u;  // slot % 8 for every slice
                float4 x, y;
#pragma unroll
                for (int j = 0; j < KS; ++j) {
                    const uint32_t row_addr = sD + static_cast<uint32_t>(j * C::KS_ROWS + r) * C::KS_ROW_BYTES;
                    const uint4 a = ptx::ld_shared_v4(row_addr + ((static_cast<uint32_t>(2 * ch) ^ sw) * 16u));
                    const uint4 b = ptx::ld_shared_v4(row_addr + ((static_cast<uint32_t>(2 * ch + 1) ^ sw) * 16u));
                    const float4 fa = make_float4(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z),
                                                  __uint_as_float(a.w));
                    const float4 fb = make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z),
                                                  __uint_as_float(b.w));
                    if (j == 0) {
                        x = fa, y = fb;
                    } else {
                        x.x += fa.x, x.y += fa.y, x.z += fa.z, x.w += fa.w;
                        y.x += fb.x, y.y += fb.y, y.z += fb.z, y.w += fb.w;
                    }
                }
                const int32_t row = o.d_row + static_cast<int32_t>(krank) * C::KS_ROWS + r;
                const int32_t col = o.d_col + 8 * ch;
                if (row < p.M && col < p.N) {
                    const __half2 h0 = __floats2half2_rn(x.x, x.y), h1 = __floats2half2_rn(x.z, x.w);
                    const __half2 h2 = __floats2half2_rn(y.x, y.y), h3 = __floats2half2_rn(y.z, y.w);
                    ptx::st_global_v4(p.D + static_cast<int64_t>(row) * p.N + col,
                                      *reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                                      *reinterpret_cast<const uint32_t *>(&h2), *reinterpret_cast<const uint32_t *>(&h3));
                }
            }
        }
        ptx::cluster_wait();
        if (warp == 1) {
            ptx::tcgen05_fence_after();
            ptx::tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
        }
        return;
    }

    // ---- teardown: the cluster's CTAs done with TMEM and with each other's
    // SMEM (the epilogue warps of a pair arrived after their last TMEM read)
    ptx::tcgen05_fence_before();
    if constexpr (C::CLUSTER > 1) {
        if (!cluster_arrived) ptx::cluster_arrive();
        ptx::cluster_wait();
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tcgen05_fence_after();
        ptx::tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
    }
}

// Split-K, second pass: D = fp16_RNE(sum over slices of the fp32 partials),
// 8 columns (16 bytes of D) per thread and step.  Launched right behind the
// GEMM as a programmatic dependent; griddepcontrol.wait makes the partials
// visible before they are read.
constexpr int kMaxSlices = 16;

template <int S>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ partial,
                                                            uint16_t *__restrict__ D, int64_t mn) {
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int64_t units = mn / 4;  // 4 columns (one float4 per slice) per thread and step
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units; u += stride) {
        // all S loads in flight before the first add; slices added in order
        float4 v[S];
#pragma unroll
        for (int s = 0; s < S; ++s) v[s] = __ldg(reinterpret_cast<const float4 *>(partial + s * mn) + u);
        float4 acc = v[0];
#pragma unroll
        for (int s = 1; s < S; ++s) {
            acc.x += v[s].x;
            acc.y += v[s].y;
            acc.z += v[s].z;
            acc.w += v[s].w;
        }
        const __half2 h0 = __floats2half2_rn(acc.x, acc.y);
        const __half2 h1 = __floats2half2_rn(acc.z, acc.w);
        *reinterpret_cast<uint2 *>(D + u * 4) =
            make_uint2(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1));
    }
}

// D = 0 for an empty contraction (K == 0): every output element is the sum of
// no products.
__global__ void zero_fill_kernel(uint4 *D, int64_t n16, uint16_t *tail, int64_t ntail) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
        D[i] = make_uint4(0, 0, 0, 0);
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < ntail; i += stride) {
        tail[i] = 0;
    }
}

}  // namespace gemm_f16
