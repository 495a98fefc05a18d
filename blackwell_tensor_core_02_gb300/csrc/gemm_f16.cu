// gemm_f16.cu -- host side of the C ABI declared in include/gemm_f16.h:
// argument validation, TMA tensor-map encoding, per-device launch caches and
// the cluster launch of the persistent kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_f16.h"
#include "gemm_kernel.cuh"
#include "schedule.h"

namespace gemm_f16 {
namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kDefaultTimeoutNs = 4000000000LL;
constexpr int64_t kDimLimit = (int64_t(1) << 31) - 1;
// Largest M, N or K a GEMM accepts: the kernel forms tile coordinates (a
// tile's first row or column plus up to 512) in 32-bit integers, and a TMA
// store must never start at a coordinate that wrapped negative.
constexpr int64_t kShapeLimit = kDimLimit - 1023;

struct DeviceInfo {
    bool ready = false;
    int status = GEMM_OK;
    int sm_count = 0;
    int max_clusters[GEMM_F16_CONFIG_KINDS] = {};  // co-resident clusters (the order of gemm_f16_co_resident):
                                // [0] cta_group 1, [1] pair, [2] pair + 2 consumers,
                                // [3] narrow single-CTA tiles, [4] tiny tiles, [5] [6] [7] tiny tiles with
                                // K split across clusters of 2, 4 and 8 CTAs, [8] [9] [10] narrow tiles
                                // likewise
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <int CG, int NC, int BN, int BM, int KS = 1>
cudaLaunchConfig_t launch_config(dim3 grid, cudaStream_t stream, cudaLaunchAttribute *attr, bool overlap = false) {
    using C = Cfg<CG, NC, BN, BM, KS>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (overlap) {
        // Programmatic dependent launch: this grid may be scheduled while the
        // previous kernel of the stream finishes; the kernel waits for it
        // (griddepcontrol.wait) before its first access to A, B or D.
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    return cfg;
}

template <int CG, int NC, int BN, int BM = 128, int KS = 1>
int prepare_kernel(int *max_clusters) {
    using C = Cfg<CG, NC, BN, BM, KS>;
    cudaError_t e = cudaFuncSetAttribute(gemm_f16_nt_kernel<CG, NC, BN, BM, KS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    if constexpr (C::REG_SPLIT) {
        // The register split (setmaxnreg) is sized for a pool of THREADS x REGS_AT_LAUNCH
        // registers: with fewer per thread, an epilogue warpgroup's increase would wait for
        // registers that never come.  A build that compiled this kernel otherwise is unusable.
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, gemm_f16_nt_kernel<CG, NC, BN, BM, KS>) != cudaSuccess ||
            fa.numRegs != C::REGS_AT_LAUNCH) {
            return GEMM_ERR_CUDA;
        }
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config<CG, NC, BN, BM, KS>(dim3(C::CLUSTER, 1, 1), nullptr, attr);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm_f16_nt_kernel<CG, NC, BN, BM, KS>, &cfg);
    if (e != cudaSuccess || n <= 0) return GEMM_ERR_CUDA;
    *max_clusters = n;
    return GEMM_OK;
}

// Per-device set-up, once: architecture check, SM count, kernel attributes,
// co-resident cluster counts, and the driver's tensor-map encoder.
int device_setup(int *dev_out, DeviceInfo **info_out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        d.ready = true;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            d.status = GEMM_ERR_NO_DEVICE;
        } else if (major != 10 || minor != 3) {
            d.status = GEMM_ERR_ARCH;
        } else {
            d.status = prepare_kernel<1, 1, 256>(&d.max_clusters[0]);
            if (d.status == GEMM_OK) d.status = prepare_kernel<2, 1, 256>(&d.max_clusters[1]);
            if (d.status == GEMM_OK) d.status = prepare_kernel<2, 2, 256>(&d.max_clusters[2]);
            if (d.status == GEMM_OK) d.status = prepare_kernel<1, 1, 64>(&d.max_clusters[3]);
            if (d.status == GEMM_OK) d.status = prepare_kernel<1, 1, 64, 64>(&d.max_clusters[4]);
            // thin 64 x 16 tiles use the tiny tiles' co-resident count (their shared
            // memory is smaller, so at least as many fit; checked here)
            int thin = 0;
            if (d.status == GEMM_OK) d.status = prepare_kernel<1, 1, 16, 64>(&thin);
            if (d.status == GEMM_OK && thin < d.max_clusters[4]) d.status = GEMM_ERR_CUDA;
            // The K splits across clusters are optional: a device that cannot
            // co-schedule clusters of that size (0 co-resident) never takes them.
            if (d.status == GEMM_OK && prepare_kernel<1, 1, 64, 64, 2>(&d.max_clusters[5]) != GEMM_OK) {
                d.max_clusters[5] = 0;
            }
            if (d.status == GEMM_OK && prepare_kernel<1, 1, 64, 64, 4>(&d.max_clusters[6]) != GEMM_OK) {
                d.max_clusters[6] = 0;
            }
            if (d.status == GEMM_OK && prepare_kernel<1, 1, 64, 64, 8>(&d.max_clusters[7]) != GEMM_OK) {
                d.max_clusters[7] = 0;
            }
            if (d.status == GEMM_OK && prepare_kernel<1, 1, 64, 128, 2>(&d.max_clusters[8]) != GEMM_OK) {
                d.max_clusters[8] = 0;
            }
            if (d.status == GEMM_OK && prepare_kernel<1, 1, 64, 128, 4>(&d.max_clusters[9]) != GEMM_OK) {
                d.max_clusters[9] = 0;
            }
            if (d.status == GEMM_OK && prepare_kernel<1, 1, 64, 128, 8>(&d.max_clusters[10]) != GEMM_OK) {
                d.max_clusters[10] = 0;
            }
        }
        if (d.status == GEMM_OK && g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                d.status = GEMM_ERR_CUDA;
            } else {
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
        }
        cudaGetLastError();
    }
    *dev_out = dev;
    *info_out = &d;
    return d.status;
}

// Row-major fp16 matrix rows x cols, tiles of box_rows x 64 columns, 128-byte
// swizzle, zero fill past the edges.
int encode_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, uint32_t box_rows) {
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t estride[2] = {1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), gdim, gstride, box,
                          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// The split-K workspace viewed as [slices][M][N] fp32, stored in 32 x 32 boxes
// with the 128-byte swizzle (each box row is 32 fp32 = 128 bytes).
int encode_partial_map(CUtensorMap *map, void *ptr, int64_t slices, int64_t M, int64_t N) {
    cuuint64_t gdim[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(slices)};
    cuuint64_t gstride[2] = {static_cast<cuuint64_t>(N) * 4, static_cast<cuuint64_t>(M) * N * 4};
    cuuint32_t box[3] = {32u, 32u, 1u};
    cuuint32_t estride[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, gdim, gstride, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

bool overlaps(const void *p, int64_t p_bytes, const void *q, int64_t q_bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + static_cast<uintptr_t>(q_bytes) && b < a + static_cast<uintptr_t>(p_bytes);
}

bool shape_ok(int64_t M, int64_t N, int64_t K) {
    return M >= 0 && N >= 0 && K >= 0 && M <= kShapeLimit && N <= kShapeLimit && K <= kShapeLimit && N % 8 == 0 &&
           K % 8 == 0;
}

struct Opts {
    int32_t cta_group = 0;  // 0: chosen from the shape (resolve_config)
    int32_t consumers = 0;  // MMA consumers 1 or 2; 0: chosen from the shape (resolve_config)
    int32_t block_n = 0;    // tile width 256, 64 or 16; 0: chosen from the shape (resolve_config)
    int32_t block_m = 0;    // rows per CTA 128 or 64 (64 only with block_n 64); 0: chosen likewise
    int32_t cluster_k = 0;  // narrow / tiny tiles: K split across clusters of 2, 4 or 8 CTAs; 1 none; 0 chosen
                            // likewise
    int32_t max_clusters = 0;
    int32_t raster_group = 0;
    int64_t timeout_ns = kDefaultTimeoutNs;
    uint32_t debug_flags = 0;
    bool overlap = true;
};

int parse_options(const gemm_f16_options *opts, Opts *o) {
    if (opts) {
        if (opts->consumers < 0 || opts->consumers > 2) return GEMM_ERR_INVALID_ARG;
        o->consumers = opts->consumers;
        if (opts->overlap_launch < -1 || opts->overlap_launch > 1) return GEMM_ERR_INVALID_ARG;
        if (opts->overlap_launch == -1) o->overlap = false;
        if (opts->cta_group != 0) o->cta_group = opts->cta_group;
        if (opts->block_n != 0 && opts->block_n != 16 && opts->block_n != 64 && opts->block_n != 256) {
            return GEMM_ERR_INVALID_ARG;
        }
        o->block_n = opts->block_n;
        if (opts->block_m != 0 && opts->block_m != 64 && opts->block_m != 128) return GEMM_ERR_INVALID_ARG;
        o->block_m = opts->block_m;
        if (opts->cluster_k != 0 && opts->cluster_k != 1 && opts->cluster_k != 2 && opts->cluster_k != 4 &&
            opts->cluster_k != 8) {
            return GEMM_ERR_INVALID_ARG;
        }
        o->cluster_k = opts->cluster_k;
        if (opts->max_clusters < 0 || opts->raster_group < 0 || opts->timeout_ns < 0 ||
            (opts->debug_flags & ~static_cast<int32_t>(kDebugProducerPhase0)) != 0) {
            return GEMM_ERR_INVALID_ARG;
        }
        o->debug_flags = static_cast<uint32_t>(opts->debug_flags);
        o->max_clusters = opts->max_clusters;
        o->raster_group = opts->raster_group;
        if (opts->timeout_ns != 0) o->timeout_ns = opts->timeout_ns;
    }
    if (o->cta_group != 0 && o->cta_group != 1 && o->cta_group != 2) return GEMM_ERR_INVALID_ARG;
    if (o->consumers == 2 && o->cta_group == 1) return GEMM_ERR_INVALID_ARG;
    if (o->block_n == 16) {
        // thin tiles: 64 rows, one CTA, one consumer, no K split
        if (o->block_m == 128 || o->cluster_k > 1 || o->cta_group == 2 || o->consumers == 2) {
            return GEMM_ERR_INVALID_ARG;
        }
        o->block_m = 64;
        o->cluster_k = 1;
        return GEMM_OK;
    }
    if (o->cluster_k > 1) {
        // the K split runs on 64-wide tiles: tiny ones unless 128 rows are asked for
        if (o->block_n == 256) return GEMM_ERR_INVALID_ARG;
        o->block_n = 64;
        if (o->block_m == 0) o->block_m = 64;
    }
    if (o->block_m == 64) {
        if (o->block_n == 256) return GEMM_ERR_INVALID_ARG;
        o->block_n = 64;  // 64-row tiles are 64 wide (or 16, the thin tiles above)
    }
    if (o->block_n == 64 && (o->cta_group == 2 || o->consumers == 2)) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

// The K split of narrow (128 x 64) and tiny (64 x 64) tiles across a cluster
// (cluster_k).  Each cluster owns one tile and each of its KS CTAs one K
// slice, so a CTA streams 1/KS of the tile's operands: small problems with a
// long K are bound by how fast one SM's loads arrive, not by the tensor pipe.
// The slices' fp32 sums meet in shared memory through the copy engine and are
// added in the same kernel (no workspace, no second launch), which costs
// about half a microsecond more than the tiles alone.  Measured on GB300 with
// tiny tiles (graph-timed, us, KS = 1 / 2 / 4 / 8): 256x256x128 2.15 / 2.70, 256x256x512 2.86 / 3.00 / 2.79 / 6.11
// (16 clusters of 8 do not all fit at once: two waves), 256x256x1024 4.12 /
// 3.55 / 3.07, 256x256x4096 10.10 / 6.81 / 4.81 / 8.15, 128x128x4096 10.13 /
// 6.64 / 4.65 / 3.49, 128x1024x1024 4.25 / 3.61 / 3.91, 384x384x2048 6.21 /
// 4.84 / 4.78, 512x512x512 2.90 / 3.87, 512x512x4096 10.25 / 8.10 / 11.97.
// So the split pays from 8 K tiles of 64 on, with at least 2 per CTA, while
// the grid leaves half of the SMs to the next kernel's set-up (tiles * KS at
// most half the co-resident CTAs); with at least 24 K tiles per CTA a whole
// wave of clusters still pays.  Tiny tiles, which stage two K tiles at a time,
// run a short K faster unsplit, so for them the split starts at 12 K tiles,
// and clusters of 8 pay only while they fill at most a quarter of the
// co-resident CTAs (graph-timed, us, KS = 1 / 2 / 4 / 8): 256x256x512 2.68 /
// 3.06 / 2.83, 256x256x640 2.79 / 3.19 / 2.86, 256x256x896 3.23 / 3.40 / 2.96,
// 128x256x1024 3.45 / 3.44 / 2.92 / 3.23, 192x192x1024 3.37 / 3.44 / 2.90 /
// 3.31, 256x128x1536 4.13 / 3.88 / 3.09 / 3.37, 128x128x1024 3.43 / 3.44 / 2.89
// / 2.85, 128x128x2048 4.84 / 4.30 / 3.19 / 3.03.  Automatic: the largest KS
// of 8, 4, 2 that meets this; a grid capped by max_clusters keeps the
// persistent tiles.
// Forced: at most the number of K tiles, and halved until the device can
// co-schedule clusters of that size.
int32_t cluster_k_slot(int32_t ks, int32_t block_m) {
    return (ks == 2 ? 5 : (ks == 4 ? 6 : 7)) + (block_m == 64 ? 0 : 3);
}

int32_t cluster_k_for(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev, const Opts &o, int32_t block_m) {
    const int64_t k_tiles = (K + 63) / 64;
    const int64_t tiles = ((M + block_m - 1) / block_m) * ((N + 63) / 64);
    const int64_t ctas = dev.max_clusters[block_m == 64 ? 4 : 3];  // co-resident single CTAs of these tiles
    int32_t ks = o.cluster_k;
    if (ks == 0) {
        const bool tiny = block_m == 64;
        if (o.max_clusters > 0 || k_tiles < (tiny ? 12 : 8)) return 1;
        const int32_t options[3] = {8, 4, 2};
        for (int i = 0; i < 3; ++i) {
            const int64_t per_cta = k_tiles / options[i];
            if (per_cta < 2 || tiles > dev.max_clusters[cluster_k_slot(options[i], block_m)]) continue;
            const int64_t share = tiny && options[i] == 8 ? 4 : 2;  // at most 1/share of the CTAs
            if (share * tiles * options[i] <= ctas || per_cta >= 24) return options[i];
        }
        return 1;
    }
    // every CTA needs a K tile, and the device must co-schedule clusters of that size
    while (ks > 1 && (ks > k_tiles || dev.max_clusters[cluster_k_slot(ks, block_m)] <= 0)) ks /= 2;
    return ks;
}

// Rows per tile and K split for a problem on 64-wide tiles (block_n 64).
// Tiny tiles when they fill at most two thirds of a wave, else narrow ones,
// each with the split cluster_k_for() gives them.  With a long K the narrow
// tiles win in two cases (measured on GB300, graph-timed, us): where the tiny
// tiles get no split but the narrow ones do with at least 16 K tiles per CTA
// (640x640x4096 10.68 -> 9.33, 768x512x4096 10.68 -> 9.24, 512x512x2048
// 6.25 -> 5.76), and where the tiny tiles split in 2 and the narrow ones can
// split in 4 with at least 8 K tiles per CTA: the same grid with a quarter
// fewer operand bytes per CTA (512x512x4096 8.09 -> 7.12, 384x384x2048
// 4.82 -> 4.41).  With a shorter K the extra exchange loses (128x1024x1024
// 3.61 -> 3.96, 512x512x1024 4.21 -> 4.66).  block_m and cluster_k given by
// the caller are kept.
void small_tiles(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev, Opts *o) {
    const int32_t forced_k = o->cluster_k;
    if (o->block_m != 0) {
        o->cluster_k = cluster_k_for(M, N, K, dev, *o, o->block_m);
        return;
    }
    int64_t ctas = dev.max_clusters[4];
    if (o->max_clusters > 0 && o->max_clusters < ctas) ctas = o->max_clusters;
    const bool tiny_fits = 3 * ((M + 63) / 64) * ((N + 63) / 64) <= 2 * ctas;
    const int32_t ks_narrow = cluster_k_for(M, N, K, dev, *o, 128);
    if (!tiny_fits) {
        o->block_m = 128;
        o->cluster_k = ks_narrow;
        return;
    }
    const int32_t ks_tiny = cluster_k_for(M, N, K, dev, *o, 64);
    const int64_t k_tiles = (K + 63) / 64;
    o->block_m = 64;
    o->cluster_k = ks_tiny;
    if (forced_k != 0) return;  // cluster_k given (1: no split): keep the tiny tiles
    if (ks_tiny == 1 && ks_narrow > 1 && k_tiles / ks_narrow >= 16) {
        o->block_m = 128;
        o->cluster_k = ks_narrow;
    } else if (ks_tiny == 2 && o->max_clusters == 0 && k_tiles / 4 >= 8) {
        const int64_t tiles_narrow = ((M + 127) / 128) * ((N + 63) / 64);
        if (tiles_narrow <= dev.max_clusters[cluster_k_slot(4, 128)] && 4 * tiles_narrow <= dev.max_clusters[3]) {
            o->block_m = 128;
            o->cluster_k = 4;
        }
    }
}

// Whether a problem whose 128 x 64 tiles fit one wave would take its narrow
// or tiny tiles with a K split (which then wins over split-K through a
// workspace: 768x768x4096 10.07 vs 12.84, 512x512x4096 7.12 vs 9.30,
// 256x256x4096 4.81 vs 8.69 us).
bool cluster_k_applies(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev, const Opts &o) {
    if (o.cluster_k == 1) return false;
    Opts t = o;
    small_tiles(M, N, K, dev, &t);
    return t.cluster_k > 1;
}

// The default CTA group and tile width.
// - A CTA pair pays a cluster handshake per stage and a cluster barrier at both
//   ends of the kernel.  That is repaid by its halved operand traffic over a
//   long K-loop, but not when the K-loop is at most 8 tiles of 64 and the pair
//   tiles would occupy at most half the pairs (measured on GB300: 128x128x64
//   2.9 vs 3.7 us, 256x256x512 5.0 vs 5.5 us single vs pair).  Such problems
//   run on single CTAs; everything else on pairs.
// - A problem whose 128 x 64 tiles fit one wave of co-resident CTAs leaves
//   most SMs idle with 256-wide tiles.  Narrow tiles spread it over up to 4x
//   as many SMs, each with a K-loop a quarter as long, and their 8-stage ring
//   holds a K of 512 at once (one load latency for a short problem).  Measured
//   on GB300 (graph-timed, us, narrow vs 256-wide): 128x128x64 2.56 vs 2.95,
//   256x256x512 3.83 vs 4.85, 1024x1024x1024 5.6 vs 6.4, 1024x1024x4096 12.1
//   vs 15.4; past one wave the 256-wide tiles win (2048x1024x512 5.7 vs 5.2).
//   With a workspace (allow_splitk), a split-K of at least 8 slices over CTA
//   pairs beats them (512x512x4096 9.8 vs 11.4, 256x256x4096 9.2 vs 11.6); 4
//   slices do not (1024x1024x4096 14.9 vs 12.1).
// - Narrow tiles whose 64 x 64 halves fill at most two thirds of a wave go
//   one step further, to 64-row tiles: twice the CTAs again, each with half
//   the MMA work per K tile.  Measured on GB300 (graph-timed, us, 64 vs 128
//   rows, tiles of 64 x 64 in brackets): 128x128x64 2.27 vs 2.53 (4),
//   512x512x512 3.47 vs 3.76 (64), 256x256x4096 10.3 vs 11.8 (16),
//   576x576x1024 5.00 vs 5.62 (81), 640x640x512 3.87 vs 3.93 (100); with more
//   the 128-row tiles win (128x4096x512 4.01 vs 3.80 and 512x1024x512 3.99
//   vs 3.77 (128), 768x768x512 4.14 vs 4.07 (144)), past one wave by far
//   (1024x1024x512 5.21 vs 4.28).
void resolve_config(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev, bool allow_splitk, Opts *o) {
    const int64_t k_tiles = (K + 63) / 64;
    // tile shape left to the library entirely (the thin tiles below are only chosen then)
    const bool auto_tile = o->block_n == 0 && o->block_m == 0 && o->cluster_k == 0;
    if (o->block_n == 16) {
        o->cta_group = 1;
        o->consumers = 1;
        return;
    }
    if (o->block_n == 0) {
        bool narrow = false;
        if (o->cta_group == 0 && o->consumers != 2) {
            int64_t ctas = dev.max_clusters[3];
            if (o->max_clusters > 0 && o->max_clusters < ctas) ctas = o->max_clusters;
            narrow = ((M + 127) / 128) * ((N + 63) / 64) <= ctas;
            if (narrow && allow_splitk && !cluster_k_applies(M, N, K, dev, *o)) {
                int64_t pairs = dev.max_clusters[1];
                if (o->max_clusters > 0 && o->max_clusters < pairs) pairs = o->max_clusters;
                const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
                if (pair_tiles <= kDimLimit && splitk_slices(static_cast<int32_t>(pair_tiles),
                                                             static_cast<int32_t>(pairs),
                                                             static_cast<int32_t>(k_tiles)) >= 8) {
                    narrow = false;
                }
            }
        }
        o->block_n = narrow ? 64 : 256;
    }
    if (o->block_n == 64) {
        o->cta_group = 1;
        o->consumers = 1;
        small_tiles(M, N, K, dev, o);
        // Thin 64 x 16 tiles for the shortest of these problems: where the tiny tiles
        // apply with a K of at most 768 (12 K tiles) and the thin tiles fill at most
        // half of the co-resident CTAs, each CTA loads and drains a quarter as much.
        // Measured on GB300 (graph-timed, us, thin vs the best other tiles): 128x128x64
        // 1.57 vs 1.76, 256x256x512 2.48 vs 2.68, 256x256x640 2.63 vs 2.79, 256x256x768
        // 2.81 vs 2.94, 128x256x768 2.83 vs 2.91; with a longer K the cluster K split
        // wins (256x256x896 3.09 vs 2.96, 128x128x1024 3.25 vs 2.85), and with more thin
        // tiles the tiny ones unsplit, whose operands cross L2 a quarter as often
        // (thin tiles in brackets: 320x256x512 2.64 vs 2.64 (80), 384x256x512 2.73 vs
        // 2.63 (96), 512x256x512 2.91 vs 2.65 (128), 384x384x256 2.55 vs 2.33 (144),
        // 384x384x64 2.11 vs 1.98 (144)).  64 x 8 tiles gained nothing more (1.60 and
        // 2.90 at 128x128x64 and 256x256x512), 64 x 32 less (1.74 and 2.83).
        int64_t ctas = dev.max_clusters[4];
        if (o->max_clusters > 0 && o->max_clusters < ctas) ctas = o->max_clusters;
        const int64_t thin_tiles = ((M + 63) / 64) * ((N + 15) / 16);
        if (auto_tile && o->block_m == 64 && k_tiles <= 12 && 2 * thin_tiles <= ctas) {
            o->block_n = 16;
            o->cluster_k = 1;
        }
        return;
    }
    o->cluster_k = 1;
    o->block_m = 128;
    if (o->consumers == 0) {
        // Two MMA consumers (512 x 256 tiles, B staged once for both) move a quarter fewer
        // operand bytes from L2 per FLOP and draw less power per clock, so under the power cap
        // they run faster; but with one accumulator per consumer the MMA waits for the
        // epilogue's TMEM reads at every tile, which only a long K-loop amortises.  Measured on
        // GB300 (graph-timed, ~1.2 s windows at the power cap, TFLOP/s, two consumers vs one):
        // K >= 6144 gains: 4096x4096x8192 1562 vs 1524, 6144^3 1613 vs 1587, 8192^3 1642 vs 1597,
        // 12288^3 1626 vs 1582, 8192x8192x16384 1638 vs 1568, 16384x8192x8192 1648 vs 1626;
        // K <= 4096 loses: 4096^3 1535 vs 1564, 8192x8192x4096 1628 vs 1643,
        // 8192x28672x4096 1662 vs 1677, 8192x8192x2048 1575 vs 1603.  So: two consumers from
        // 96 K tiles of 64 on, when their tiles fill at least one wave of co-resident pairs.
        int64_t pairs = dev.max_clusters[2];
        if (o->max_clusters > 0 && o->max_clusters < pairs) pairs = o->max_clusters;
        const int64_t tiles2 = ((M + 511) / 512) * ((N + 255) / 256);
        o->consumers = (o->cta_group != 1 && k_tiles >= 96 && tiles2 >= pairs) ? 2 : 1;
    }
    if (o->cta_group != 0) return;
    if (o->consumers == 2) {
        o->cta_group = 2;
        return;
    }
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    int64_t pairs = dev.max_clusters[1];
    if (o->max_clusters > 0 && o->max_clusters < pairs) pairs = o->max_clusters;
    o->cta_group = (k_tiles <= 8 && 2 * pair_tiles <= pairs) ? 1 : 2;
}

// Everything about one launch that follows from the shape, the options and
// the device: tile counts, scheduler parameters, split-K slices, grid size.
struct Plan {
    Params p;
    int64_t clusters;          // persistent clusters launched
    int64_t workspace_bytes;   // split-K partials, 0 without split-K
};

template <int CG, int NC, int BN, int BM = 128, int KS = 1>
int make_plan(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev, const Opts &o, bool allow_splitk,
              Plan *out) {
    using C = Cfg<CG, NC, BN, BM, KS>;
    Params &p = out->p;
    p = Params{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.num_m_tiles = static_cast<int32_t>((M + C::TILE_M - 1) / C::TILE_M);
    p.num_n_tiles = static_cast<int32_t>((N + C::BLOCK_N - 1) / C::BLOCK_N);
    p.k_tiles = static_cast<int32_t>((K + C::BLOCK_K - 1) / C::BLOCK_K);
    const int64_t tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
    if (tiles > kDimLimit / 16) return GEMM_ERR_UNSUPPORTED_SHAPE;
    p.num_tiles = static_cast<int32_t>(tiles);
    p.raster_group = o.raster_group > 0 ? o.raster_group : auto_raster_group(p.num_m_tiles, K, C::TILE_M);
    p.debug_flags = o.debug_flags;
    p.timeout_ns = static_cast<uint64_t>(o.timeout_ns);
    if constexpr (C::KSPLIT) {
        // one cluster per tile, CTA s of the cluster on K slice s: item
        // t * KS + s, the numbering of split-K, one item per CTA
        p.slices = KS;
        p.split_from = p.num_tiles;
        p.num_items = p.num_tiles * KS;
        out->workspace_bytes = 0;
        out->clusters = p.num_tiles;
        return GEMM_OK;
    }
    int64_t clusters = dev.max_clusters[C::KIND];
    if (o.max_clusters > 0 && o.max_clusters < clusters) clusters = o.max_clusters;
    p.slices = (allow_splitk && NC == 1 && !C::NARROW)
                   ? splitk_slices(p.num_tiles, static_cast<int32_t>(clusters), p.k_tiles)
                   : 1;
    if (p.slices > kMaxSlices) p.slices = kMaxSlices;
    if (p.slices > 1) {
        p.split_from = p.num_tiles;
        p.num_items = p.num_tiles * p.slices;
        out->workspace_bytes = static_cast<int64_t>(p.slices) * M * N * static_cast<int64_t>(sizeof(float));
    } else {
        // narrow tiles are not split along N: a 32-column half would leave
        // the MMA bound by its A operand reads
        p.split_from = C::NARROW ? p.num_tiles : split_point(p.num_tiles, static_cast<int32_t>(clusters));
        p.num_items = p.num_tiles + (p.num_tiles - p.split_from);
        out->workspace_bytes = 0;
    }
    if (clusters > p.num_items) clusters = p.num_items;
    out->clusters = clusters;
    return GEMM_OK;
}

template <int S>
cudaError_t launch_reduce_s(const cudaLaunchConfig_t *cfg, const float *partial, uint16_t *D, int64_t mn) {
    return cudaLaunchKernelEx(cfg, splitk_reduce_kernel<S>, partial, D, mn);
}

cudaError_t launch_reduce(const cudaLaunchConfig_t *cfg, int slices, const float *partial, uint16_t *D, int64_t mn) {
    switch (slices) {
        case 4: return launch_reduce_s<4>(cfg, partial, D, mn);
        case 5: return launch_reduce_s<5>(cfg, partial, D, mn);
        case 6: return launch_reduce_s<6>(cfg, partial, D, mn);
        case 7: return launch_reduce_s<7>(cfg, partial, D, mn);
        case 8: return launch_reduce_s<8>(cfg, partial, D, mn);
        case 9: return launch_reduce_s<9>(cfg, partial, D, mn);
        case 10: return launch_reduce_s<10>(cfg, partial, D, mn);
        case 11: return launch_reduce_s<11>(cfg, partial, D, mn);
        case 12: return launch_reduce_s<12>(cfg, partial, D, mn);
        case 13: return launch_reduce_s<13>(cfg, partial, D, mn);
        case 14: return launch_reduce_s<14>(cfg, partial, D, mn);
        case 15: return launch_reduce_s<15>(cfg, partial, D, mn);
        case 16: return launch_reduce_s<16>(cfg, partial, D, mn);
        default: return cudaErrorInvalidValue;
    }
}

template <int CG, int NC, int BN, int BM = 128, int KS = 1>
int launch(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
           const DeviceInfo &dev, const Opts &o, void *workspace, int64_t workspace_bytes) {
    using C = Cfg<CG, NC, BN, BM, KS>;
    Plan plan;
    int st = make_plan<CG, NC, BN, BM, KS>(M, N, K, dev, o, workspace != nullptr, &plan);
    if (st != GEMM_OK) return st;
    if (plan.p.slices > 1 && !C::KSPLIT &&
        (workspace_bytes < plan.workspace_bytes || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)) {
        st = make_plan<CG, NC, BN, BM, KS>(M, N, K, dev, o, false, &plan);  // workspace too small: no split-K
        if (st != GEMM_OK) return st;
    }
    Params &p = plan.p;
    CUtensorMap tmA, tmB, tmBh, tmD;
    if (encode_map(&tmA, A, M, K, C::BLOCK_M) != GEMM_OK || encode_map(&tmB, B, N, K, C::B_ROWS) != GEMM_OK ||
        encode_map(&tmBh, B, N, K, C::B_ROWS / 2) != GEMM_OK || encode_map(&tmD, D, M, N, 32) != GEMM_OK) {
        return GEMM_ERR_CUDA;
    }
    p.D = reinterpret_cast<uint16_t *>(D);
    p.partial = p.slices > 1 && !C::KSPLIT ? reinterpret_cast<float *>(workspace) : nullptr;
    CUtensorMap tmP;
    if (p.slices > 1 && !C::KSPLIT) {
        if (encode_partial_map(&tmP, workspace, p.slices, M, N) != GEMM_OK) return GEMM_ERR_CUDA;
    } else {
        tmP = tmD;  // unused without split-K
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config<CG, NC, BN, BM, KS>(
        dim3(static_cast<unsigned>(plan.clusters * C::CLUSTER), 1, 1), stream, attr, o.overlap);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_f16_nt_kernel<CG, NC, BN, BM, KS>, tmA, tmB, tmBh, tmD, tmP, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (p.slices > 1 && !C::KSPLIT) {
        // second pass: add the slices' partials and round once (its CTAs may
        // start early; griddepcontrol.wait orders it after the GEMM)
        const int64_t units = M * N / 4;
        int64_t blocks = (units + 255) / 256;
        if (blocks > 8 * dev.sm_count) blocks = 8 * dev.sm_count;
        if (blocks < 1) blocks = 1;
        cudaLaunchConfig_t rcfg = {};
        rcfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
        rcfg.blockDim = dim3(256, 1, 1);
        rcfg.stream = stream;
        cudaLaunchAttribute rattr[1];
        rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        rattr[0].val.programmaticStreamSerializationAllowed = 1;
        rcfg.attrs = rattr;
        rcfg.numAttrs = 1;
        e = launch_reduce(&rcfg, p.slices, static_cast<const float *>(p.partial), reinterpret_cast<uint16_t *>(D),
                          M * N);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    }
    return GEMM_OK;
}

int zero_fill(void *D, int64_t M, int64_t N, cudaStream_t stream);

// The argument checks every compute entry point makes before anything is enqueued (A, B, D
// are the device operands).  GEMM_OK also for an empty product, which then launches nothing.
int check_args(const void *A, const void *B, const void *D, int64_t M, int64_t N, int64_t K,
               const gemm_f16_options *opts, Opts *o) {
    int st = parse_options(opts, o);
    if (st != GEMM_OK) return st;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (!shape_ok(M, N, K)) return GEMM_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return GEMM_OK;  // empty product: nothing to write
    if (!D || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(D) & 15u) || (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15u) ||
                                                             (reinterpret_cast<uintptr_t>(B) & 15u)))) {
        return GEMM_ERR_MISALIGNED;
    }
    // D is written while A and B are still being read: their byte ranges must not meet
    if (K > 0 && (overlaps(D, M * N * 2, A, M * K * 2) || overlaps(D, M * N * 2, B, N * K * 2))) {
        return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

int run(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *stream,
        const gemm_f16_options *opts, void *workspace, int64_t workspace_bytes) {
    Opts o;
    if (workspace_bytes < 0) return GEMM_ERR_INVALID_ARG;
    int st = check_args(A, B, D, M, N, K, opts, &o);
    if (st != GEMM_OK || M == 0 || N == 0) return st;
    int dev = -1;
    DeviceInfo *info = nullptr;
    st = device_setup(&dev, &info);
    if (st != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return zero_fill(D, M, N, s);
    resolve_config(M, N, K, *info, workspace != nullptr, &o);
    if (o.block_n == 16) return launch<1, 1, 16, 64>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
    if (o.block_n == 64 && o.block_m == 64) {
        switch (o.cluster_k) {
            case 2: return launch<1, 1, 64, 64, 2>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
            case 4: return launch<1, 1, 64, 64, 4>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
            case 8: return launch<1, 1, 64, 64, 8>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
            default: return launch<1, 1, 64, 64>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
        }
    }
    if (o.block_n == 64) {
        switch (o.cluster_k) {
            case 2: return launch<1, 1, 64, 128, 2>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
            case 4: return launch<1, 1, 64, 128, 4>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
            case 8: return launch<1, 1, 64, 128, 8>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
            default: return launch<1, 1, 64>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
        }
    }
    if (o.cta_group == 2 && o.consumers == 2) return launch<2, 2, 256>(A, B, D, M, N, K, s, *info, o, nullptr, 0);
    if (o.cta_group == 2) return launch<2, 1, 256>(A, B, D, M, N, K, s, *info, o, workspace, workspace_bytes);
    return launch<1, 1, 256>(A, B, D, M, N, K, s, *info, o, workspace, workspace_bytes);
}

// What a call would launch on a device with these co-resident cluster counts
// (the body of gemm_f16_nt_describe and gemm_f16_nt_describe_for).
int describe_with(const DeviceInfo &info, Opts o, int64_t M, int64_t N, int64_t K, bool ws,
                  gemm_f16_launch_info *out) {
    int st = GEMM_OK;
    resolve_config(M, N, K, info, ws, &o);
    Plan plan;
    int stages = 0;
    if (o.block_n == 16) {
        st = make_plan<1, 1, 16, 64>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 16, 64>::STAGES * Cfg<1, 1, 16, 64>::KPS;
    } else if (o.block_n == 64 && o.block_m == 64 && o.cluster_k == 2) {
        st = make_plan<1, 1, 64, 64, 2>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64, 64, 2>::STAGES * Cfg<1, 1, 64, 64, 2>::KPS;
    } else if (o.block_n == 64 && o.block_m == 64 && o.cluster_k == 4) {
        st = make_plan<1, 1, 64, 64, 4>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64, 64, 4>::STAGES * Cfg<1, 1, 64, 64, 4>::KPS;
    } else if (o.block_n == 64 && o.block_m == 64 && o.cluster_k == 8) {
        st = make_plan<1, 1, 64, 64, 8>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64, 64, 8>::STAGES * Cfg<1, 1, 64, 64, 8>::KPS;
    } else if (o.block_n == 64 && o.block_m == 64) {
        st = make_plan<1, 1, 64, 64>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64, 64>::STAGES * Cfg<1, 1, 64, 64>::KPS;
    } else if (o.block_n == 64 && o.cluster_k == 2) {
        st = make_plan<1, 1, 64, 128, 2>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64, 128, 2>::STAGES * Cfg<1, 1, 64, 128, 2>::KPS;
    } else if (o.block_n == 64 && o.cluster_k == 4) {
        st = make_plan<1, 1, 64, 128, 4>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64, 128, 4>::STAGES * Cfg<1, 1, 64, 128, 4>::KPS;
    } else if (o.block_n == 64 && o.cluster_k == 8) {
        st = make_plan<1, 1, 64, 128, 8>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64, 128, 8>::STAGES * Cfg<1, 1, 64, 128, 8>::KPS;
    } else if (o.block_n == 64) {
        st = make_plan<1, 1, 64>(M, N, K, info, o, false, &plan);
        stages = Cfg<1, 1, 64>::STAGES * Cfg<1, 1, 64>::KPS;
    } else if (o.cta_group == 2 && o.consumers == 2) {
        st = make_plan<2, 2, 256>(M, N, K, info, o, false, &plan);
        stages = Cfg<2, 2, 256>::STAGES * Cfg<2, 2, 256>::KPS;
    } else if (o.cta_group == 2) {
        st = make_plan<2, 1, 256>(M, N, K, info, o, ws, &plan);
        stages = Cfg<2, 1, 256>::STAGES * Cfg<2, 1, 256>::KPS;
    } else {
        st = make_plan<1, 1, 256>(M, N, K, info, o, ws, &plan);
        stages = Cfg<1, 1, 256>::STAGES * Cfg<1, 1, 256>::KPS;
    }
    if (st != GEMM_OK) return st;
    out->cta_group = o.cta_group;
    out->consumers = o.consumers;
    out->block_n = o.block_n;
    out->block_m = o.block_m;
    out->stages = stages;
    out->cluster_k = o.cluster_k > 1 ? o.cluster_k : 1;
    out->split_k = o.cluster_k > 1 ? 1 : plan.p.slices;
    out->clusters = plan.clusters;
    out->work_items = plan.p.num_items;
    out->workspace_bytes = plan.workspace_bytes;
    return GEMM_OK;
}

int zero_fill(void *D, int64_t M, int64_t N, cudaStream_t stream) {
    const int64_t elems = M * N;
    const int64_t n16 = elems / 8;
    const int64_t ntail = elems - n16 * 8;
    uint16_t *tail = reinterpret_cast<uint16_t *>(D) + n16 * 8;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 65535) blocks = 65535;
    zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<uint4 *>(D), n16, tail,
                                                                         ntail);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

}  // namespace
}  // namespace gemm_f16

using namespace gemm_f16;

extern "C" {

int gemm_f16_nt_supported(int64_t M, int64_t N, int64_t K) { return shape_ok(M, N, K) ? 1 : 0; }

int gemm_f16_nt_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *stream,
                   const gemm_f16_options *opts) {
    return run(A, B, D, M, N, K, stream, opts, nullptr, 0);
}

int gemm_f16_nt(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *stream) {
    return run(A, B, D, M, N, K, stream, nullptr, nullptr, 0);
}

int gemm_f16_nt_host(const void *A_host, const void *B_host, void *D_host, int64_t M, int64_t N, int64_t K,
                     void *A_dev, void *B_dev, void *D_dev, void *stream, const gemm_f16_options *opts) {
    Opts o;
    int st = check_args(A_dev, B_dev, D_dev, M, N, K, opts, &o);
    if (st != GEMM_OK || M == 0 || N == 0) return st;
    if (!D_host || (K > 0 && (!A_host || !B_host))) return GEMM_ERR_INVALID_ARG;
    int dev = -1;
    DeviceInfo *info = nullptr;
    st = device_setup(&dev, &info);  // a usable GB300 before any copy is enqueued
    if (st != GEMM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K > 0 && (cudaMemcpyAsync(A_dev, A_host, static_cast<size_t>(M * K * 2), cudaMemcpyHostToDevice, s) !=
                      cudaSuccess ||
                  cudaMemcpyAsync(B_dev, B_host, static_cast<size_t>(N * K * 2), cudaMemcpyHostToDevice, s) !=
                      cudaSuccess)) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    st = run(A_dev, B_dev, D_dev, M, N, K, stream, opts, nullptr, 0);
    if (st != GEMM_OK) return st;
    if (cudaMemcpyAsync(D_host, D_dev, static_cast<size_t>(M * N * 2), cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

int gemm_f16_nt_ws(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *workspace,
                   int64_t workspace_bytes, void *stream, const gemm_f16_options *opts) {
    if (!workspace && workspace_bytes != 0) return GEMM_ERR_INVALID_ARG;
    return run(A, B, D, M, N, K, stream, opts, workspace, workspace_bytes);
}

int64_t gemm_f16_nt_workspace_size(int64_t M, int64_t N, int64_t K, const gemm_f16_options *opts) {
    Opts o;
    int st = parse_options(opts, &o);
    if (st != GEMM_OK) return st;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (!shape_ok(M, N, K)) return GEMM_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0 || K == 0 || o.consumers == 2) return 0;
    int dev = -1;
    DeviceInfo *info = nullptr;
    st = device_setup(&dev, &info);
    if (st != GEMM_OK) return st;
    Plan plan;
    resolve_config(M, N, K, *info, true, &o);
    if (o.block_n != 256 || o.consumers == 2) return 0;  // narrow, tiny, thin tiles and two consumers never split K
    st = o.cta_group == 2 ? make_plan<2, 1, 256>(M, N, K, *info, o, true, &plan)
                          : make_plan<1, 1, 256>(M, N, K, *info, o, true, &plan);
    if (st != GEMM_OK) return st;
    return plan.workspace_bytes;
}

int gemm_f16_nt_describe(int64_t M, int64_t N, int64_t K, const gemm_f16_options *opts, int32_t with_workspace,
                         gemm_f16_launch_info *out) {
    Opts o;
    int st = parse_options(opts, &o);
    if (st != GEMM_OK) return st;
    if (M < 0 || N < 0 || K < 0 || !out || (with_workspace != 0 && with_workspace != 1)) return GEMM_ERR_INVALID_ARG;
    if (!shape_ok(M, N, K)) return GEMM_ERR_UNSUPPORTED_SHAPE;
    *out = gemm_f16_launch_info{};
    if (M == 0 || N == 0 || K == 0) return GEMM_OK;
    int dev = -1;
    DeviceInfo *info = nullptr;
    st = device_setup(&dev, &info);
    if (st != GEMM_OK) return st;
    return describe_with(*info, o, M, N, K, with_workspace != 0, out);
}

int gemm_f16_co_resident(int32_t *out, int32_t count) {
    if (!out || count != GEMM_F16_CONFIG_KINDS) return GEMM_ERR_INVALID_ARG;
    int dev = -1;
    DeviceInfo *info = nullptr;
    const int st = device_setup(&dev, &info);
    if (st != GEMM_OK) return st;
    for (int i = 0; i < GEMM_F16_CONFIG_KINDS; ++i) out[i] = info->max_clusters[i];
    return GEMM_OK;
}

int gemm_f16_nt_describe_for(int64_t M, int64_t N, int64_t K, const gemm_f16_options *opts, int32_t with_workspace,
                             const int32_t *co_resident, int32_t count, gemm_f16_launch_info *out) {
    Opts o;
    int st = parse_options(opts, &o);
    if (st != GEMM_OK) return st;
    if (M < 0 || N < 0 || K < 0 || !out || (with_workspace != 0 && with_workspace != 1) || !co_resident ||
        count != GEMM_F16_CONFIG_KINDS) {
        return GEMM_ERR_INVALID_ARG;
    }
    DeviceInfo info;
    info.ready = true;
    for (int i = 0; i < GEMM_F16_CONFIG_KINDS; ++i) {
        // the five base configurations must run; the K splits may be missing (0)
        if (co_resident[i] < (i < 5 ? 1 : 0)) return GEMM_ERR_INVALID_ARG;
        info.max_clusters[i] = co_resident[i];
    }
    if (!shape_ok(M, N, K)) return GEMM_ERR_UNSUPPORTED_SHAPE;
    *out = gemm_f16_launch_info{};
    if (M == 0 || N == 0 || K == 0) return GEMM_OK;
    return describe_with(info, o, M, N, K, with_workspace != 0, out);
}

int gemm_f16_last_device_status(void *stream, uint64_t *info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    int status = 0;
    unsigned long long where = 0;
    const int zero = 0;
    const unsigned long long zero64 = 0;
    if (cudaMemcpyFromSymbol(&status, g_status, sizeof(int)) != cudaSuccess ||
        cudaMemcpyFromSymbol(&where, g_info, sizeof(where)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_info, &zero64, sizeof(zero64)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (info) *info = where;
    return status;
}

const char *gemm_f16_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: null pointer, negative size or bad option";
        case GEMM_ERR_UNSUPPORTED_SHAPE:
            return "GEMM_ERR_UNSUPPORTED_SHAPE: N and K must be multiples of 8, and M, N, K at most 2^31 - 1024";
        case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED: A, B and D must be 16-byte aligned";
        case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE: no usable CUDA device";
        case GEMM_ERR_ARCH: return "GEMM_ERR_ARCH: the current device is not sm_103 (GB300)";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch failed";
        case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT: a wait inside the kernel ran out";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA runtime or driver error";
        case GEMM_ERR_DEVICE_BOUNDS:
            return "GEMM_ERR_DEVICE_BOUNDS: a range check inside the kernel failed (checked build)";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "GEMM_ERR_SCRATCH_LIMIT: the split-K scratch this problem needs exceeds the library's fixed "
                   "16 MiB scratch array (use gemm_f16_nt_ws with a larger workspace)";
        default: return "unknown gemm_f16 status";
    }
}

int gemm_f16_nt_schedule(int64_t M, int64_t N, int64_t K, int32_t cta_group, int32_t consumers, int32_t block_n,
                         int32_t block_m, int32_t raster_group, int32_t split_k, int64_t num_clusters,
                         int64_t cluster_id, int64_t iter, gemm_f16_work_item *out) {
    if (block_m == 0) block_m = block_n == 16 ? 64 : 128;
    if (block_n == 0) block_n = block_m == 64 ? 64 : 256;
    if (cta_group == 0) cta_group = block_n == 256 ? 2 : 1;
    if (consumers == 0) consumers = 1;
    if ((cta_group != 1 && cta_group != 2) || (consumers != 1 && consumers != 2) ||
        (consumers == 2 && cta_group != 2) || (block_n != 16 && block_n != 64 && block_n != 256) ||
        (block_n != 256 && (cta_group != 1 || consumers != 1)) || (block_m != 64 && block_m != 128) ||
        (block_m == 64 && block_n == 256) || (block_n == 16 && block_m != 64) || raster_group < 0 ||
        (split_k != 0 && split_k != 1 && split_k != 2 && split_k != 4 && split_k != 8) ||
        (split_k > 1 && block_n != 64) || K < 0 ||
        K > kDimLimit || M <= 0 || N <= 0 || M > kDimLimit || N > kDimLimit || num_clusters <= 0 ||
        num_clusters > kDimLimit || cluster_id < 0 || cluster_id >= num_clusters || iter < 0 || !out) {
        return GEMM_ERR_INVALID_ARG;
    }
    const int64_t tile_m = int64_t(block_m) * cta_group * consumers, tile_n = block_n;
    const int64_t num_m = (M + tile_m - 1) / tile_m, num_n = (N + tile_n - 1) / tile_n;
    const int64_t tiles = num_m * num_n;
    if (tiles > kDimLimit / 16) return GEMM_ERR_INVALID_ARG;
    const int32_t k_tiles = static_cast<int32_t>((K + 63) / 64);
    if (raster_group == 0) raster_group = auto_raster_group(static_cast<int32_t>(num_m), K, static_cast<int32_t>(tile_m));
    const bool narrow = block_n != 256;
    int32_t slices = 1;
    if (split_k > 1) {
        // narrow or tiny tiles with K split across clusters of split_k CTAs (cluster_k)
        slices = split_k;
        while (slices > 1 && slices > k_tiles) slices /= 2;
    } else if (split_k && consumers == 1 && !narrow) {
        slices = splitk_slices(static_cast<int32_t>(tiles), static_cast<int32_t>(num_clusters), k_tiles);
    }
    int32_t split_from;
    int64_t items;
    if (slices > 1) {
        split_from = static_cast<int32_t>(tiles);
        items = tiles * slices;
    } else {
        split_from = narrow ? static_cast<int32_t>(tiles)
                            : split_point(static_cast<int32_t>(tiles), static_cast<int32_t>(num_clusters));
        items = tiles + (tiles - split_from);
    }
    const int64_t item = cluster_id + iter * num_clusters;
    if (item >= items) return 0;
    const WorkItem w = work_of(static_cast<int32_t>(item), static_cast<int32_t>(num_m), static_cast<int32_t>(num_n),
                               raster_group, split_from, k_tiles, slices, block_n);
    out->m_idx = w.m_idx;
    out->n_idx = w.n_idx;
    out->n_off = w.n_off;
    out->n_len = w.n_len;
    out->slice = w.slice;
    out->kt_begin = w.kt_begin;
    out->kt_end = w.kt_end;
    return 1;
}

int gemm_f16_nt_cta_origin(int32_t cta_group, int32_t consumers, int32_t block_n, int32_t block_m, int64_t m_idx,
                           int64_t n_idx, int64_t n_off, int64_t n_len, int32_t rank, int64_t *a_row, int64_t *b_row,
                           int64_t *d_row, int64_t *d_col) {
    if (block_m == 0) block_m = block_n == 16 ? 64 : 128;
    if (block_n == 0) block_n = block_m == 64 ? 64 : 256;
    if (cta_group == 0) cta_group = block_n == 256 ? 2 : 1;
    if (consumers == 0) consumers = 1;
    const bool lens_ok = block_n != 256 ? (n_len == block_n && n_off == 0)
                                        : ((n_len == 256 && n_off == 0) || (n_len == 128 && (n_off == 0 || n_off == 128)));
    if ((cta_group != 1 && cta_group != 2) || (consumers != 1 && consumers != 2) ||
        (consumers == 2 && cta_group != 2) || (block_n != 16 && block_n != 64 && block_n != 256) ||
        (block_n != 256 && (cta_group != 1 || consumers != 1)) || (block_m != 64 && block_m != 128) ||
        (block_m == 64 && block_n == 256) || (block_n == 16 && block_m != 64) || rank < 0 || rank >= cta_group ||
        m_idx < 0 || n_idx < 0 ||
        m_idx * block_m * cta_group * consumers > kDimLimit || n_idx * block_n > kDimLimit || !lens_ok ||
        !a_row || !b_row || !d_row || !d_col) {
        return GEMM_ERR_INVALID_ARG;
    }
    WorkItem w;
    w.m_idx = static_cast<int32_t>(m_idx);
    w.n_idx = static_cast<int32_t>(n_idx);
    w.n_off = static_cast<int32_t>(n_off);
    w.n_len = static_cast<int32_t>(n_len);
    const CtaOrigin o = cta_origin(w, cta_group, rank, consumers, block_n, block_m);
    *a_row = o.a_row;
    *b_row = o.b_row;
    *d_row = o.d_row;
    *d_col = o.d_col;
    return GEMM_OK;
}

int gemm_f16_pipeline_trace(int32_t depth, int32_t initial_phase, int32_t steps, int32_t *stage_out,
                            int32_t *phase_out) {
    if (depth < 1 || depth > 16 || (initial_phase != 0 && initial_phase != 1) || steps < 0 ||
        (steps > 0 && (!stage_out || !phase_out))) {
        return GEMM_ERR_INVALID_ARG;
    }
    PipelineState ring(depth, static_cast<uint32_t>(initial_phase));
    for (int32_t i = 0; i < steps; ++i) {
        stage_out[i] = ring.stage;
        phase_out[i] = static_cast<int32_t>(ring.phase);
        ring.advance();
    }
    return GEMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// A GEMM entry point that allocates nothing: the split-K scratch lives in a
// fixed device array of this library instead of memory the caller provides.
//
// Who needs it: code that must not allocate device memory while it runs --
// for example a caller that sets its memory budget up front and forbids any
// later allocation, a plug-in that lives inside a host application owning all
// of the GPU's memory, or a real-time loop where an allocation (which can
// block and synchronise the device) is not allowed.  Such callers can still
// get split-K by using this fixed array.
//
// Cost: every GPU on which this library's device code is loaded holds the
// array (kStaticScratchBytes) until the process exits.  All calls on a device
// share it, and it keeps whatever the last call wrote; split-K overwrites
// every partial it later reads, so nothing in it has to start at zero, but
// two calls that may run at the same time on the GPU (different streams
// without ordering, or concurrent host threads) race on it.
// ---------------------------------------------------------------------------
namespace gemm_f16 {
namespace {

// the size the public header promises (GEMM_F16_STATIC_SCRATCH_BYTES), which is also the
// refusal limit of gemm_f16_nt_static_ws
constexpr int64_t kStaticScratchBytes = GEMM_F16_STATIC_SCRATCH_BYTES;
static_assert(kStaticScratchBytes % 256 == 0, "whole 256-byte units");

static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];

std::mutex g_static_mutex;
void *g_static_ptr[kMaxDevices] = {};

// The array's device address on the current device.  In host code the name
// g_static_scratch is only a host-side handle, never a device address, so it
// is resolved once per device, with that device current.
int static_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return GEMM_OK;
}

}  // namespace
}  // namespace gemm_f16

extern "C" int gemm_f16_nt_static_ws(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                                     void *stream, const gemm_f16_options *opts) {
    const int64_t need = gemm_f16_nt_workspace_size(M, N, K, opts);
    if (need < 0) return static_cast<int>(need);
    if (need > kStaticScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const int st = static_scratch(&scratch);
    if (st != GEMM_OK) return st;
    return gemm_f16_nt_ws(A, B, D, M, N, K, scratch, kStaticScratchBytes, stream, opts);
}
