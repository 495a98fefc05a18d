/*
 * gemm_f16.h -- C ABI of a GB300 (sm_103a) fp16 GEMM:  D = A * B^T
 *
 * The operation ("GEMM I -- the tiled baseline", section "The problem we are
 * solving"; "TIRx GEMM detailed technical notes", V8 "Operand Partition"):
 *
 *     A is M x K, B is N x K, D is M x N, all row-major, dense, IEEE binary16.
 *     D[m][n] = fp16( sum_{k<K} A[m][k] * B[n][k] )
 *
 * B is stored N x K on purpose: a row-band of B is a column-band of B^T, so
 * both operands stream as K-major row-bands.  Products and the running sum are
 * fp32 on the tensor cores (tcgen05, accumulator in tensor memory); the sum is
 * rounded to fp16 once, round-to-nearest-even, at writeback (Step 1, "round
 * once, at the end").
 *
 * Conventions shared by every call below:
 *   - Pointers named A, B, D are DEVICE pointers owned by the caller.  The
 *     library never frees, keeps or reallocates them and allocates no device
 *     memory per call.  D must not overlap A or B (a call where it does is
 *     refused with GEMM_ERR_INVALID_ARG).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Compute calls are asynchronous: they validate, enqueue their
 *     kernel on `stream` (two with split-K, the GEMM and the reduction; a fill
 *     of D with zeros when K is 0) and return; D is ready when the stream
 *     reaches that point.
 *   - Errors are negative gemm_status_t values.  An argument error is reported
 *     before anything is enqueued and leaves D untouched.  A failure inside a
 *     running kernel (a bounded wait that ran out) is reported by
 *     gemm_f16_last_device_status(), never by a hang or a trap.
 *   - Calls on different streams may run concurrently from several host
 *     threads.  The device status word is one per device, last writer wins.
 */
#ifndef GEMM_F16_H
#define GEMM_F16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad option  */
    GEMM_ERR_UNSUPPORTED_SHAPE = -2, /* see gemm_f16_nt_supported()             */
    GEMM_ERR_MISALIGNED = -3,        /* A, B or D not 16-byte aligned           */
    GEMM_ERR_NO_DEVICE = -4,         /* no CUDA device / driver usable          */
    GEMM_ERR_ARCH = -5,              /* current device is not sm_103 (GB300)    */
    GEMM_ERR_LAUNCH = -6,            /* the kernel launch itself failed         */
    GEMM_ERR_DEVICE_TIMEOUT = -7,    /* a bounded wait inside the kernel ran out */
    GEMM_ERR_CUDA = -8,              /* another CUDA runtime/driver error        */
    GEMM_ERR_SCRATCH_LIMIT = -9,     /* gemm_f16_nt_static_ws: scratch too small  */
    GEMM_ERR_DEVICE_BOUNDS = -10     /* checked build only: a device range check failed */
} gemm_status_t;

/*
 * Options for gemm_f16_nt_ex().  Zero-initialise and set what you need; every
 * zero field means "the default".
 *   cta_group     2: a 2-CTA cluster issues one cta_group::2 MMA over a
 *                 256 x 256 tile per CTA pair ("GEMM III -- warp
 *                 specialization & clusters to SOTA", Step 8; TIRx notes V8).
 *                 1: each CTA computes a 128 x 256 tile alone (Step 7 / V7).
 *                 0 (default): 1 when the K-loop is at most 8 tiles of 64 and
 *                 the pair tiles would occupy at most half the co-resident
 *                 pairs (small, latency-bound problems), else 2.  With both
 *                 cta_group and block_n at 0, small problems may instead take
 *                 the narrow tiles of block_n 64 (and the smallest the tiny
 *                 tiles of block_m 64).
 *   max_clusters  cap on the persistent grid, in clusters (CTA pairs for
 *                 cta_group 2); 0 = as many as are co-resident on the device.
 *   raster_group  L2 grouping of the tile scheduler, in M-tiles (TIRx notes
 *                 V6, "l2_group_size"); inside a group M varies fastest, and
 *                 odd groups walk N backwards (a serpentine, so a group starts
 *                 on the B panels the previous one ended on).  0 = chosen from
 *                 the shape: the largest group whose A panel (group x the
 *                 tile's rows x K fp16) fits in 32 MiB, between 1 and the
 *                 number of M-tiles.
 *   debug_flags   test hook, 0 in normal use.  1 starts the producer end of
 *                 the SMEM ring at phase 0 instead of 1 -- the pages' "subtlest
 *                 bug" ("GEMM III", "opposite initial phases") -- so that every
 *                 wait runs out; it exists to test the timeout path, which
 *                 must end the kernel with GEMM_ERR_DEVICE_TIMEOUT, not hang.
 *                 Other bits: GEMM_ERR_INVALID_ARG.
 *   timeout_ns    limit of every wait inside the kernel; 0 = 4 s.
 *   overlap_launch  0 or 1 (default): launch as a programmatic dependent of
 *                 the previous kernel on the stream, so that this kernel's
 *                 set-up (barriers, tensor memory) overlaps that kernel's
 *                 tail; the kernel still waits for it to finish, and for its
 *                 writes to be visible, before it reads A or B or writes D.
 *                 -1: an ordinary launch.  Other values: GEMM_ERR_INVALID_ARG.
 *   consumers     1: one MMA consumer per CTA pair, 256 x 256 tiles, two
 *                 accumulator buffers in tensor memory so the epilogue
 *                 overlaps the next tile.  2 (needs cta_group 0 or 2): two
 *                 consumers share each staged B tile, 512 x 256 tiles
 *                 ("GEMM III", Step 9; TIRx notes V9), one accumulator per
 *                 consumer, registers moved from the producer and MMA warps
 *                 to the epilogue warps (Step 7, setmaxnreg) so the
 *                 accumulator goes back to the MMA before D is stored.
 *                 0 (default): 2 when the K-loop is at least 96 tiles of 64
 *                 and the 512 x 256 tiles fill at least one wave of
 *                 co-resident pairs (and cta_group is not 1, block_n not
 *                 64), else 1: a long K-loop amortises the wait for the
 *                 epilogue at every tile, and the shared B tile moves a
 *                 quarter fewer operand bytes, which under the power cap
 *                 buys clock.  Other values: GEMM_ERR_INVALID_ARG.
 *   block_n       tile width in columns of D.  256: the tiles above.  64
 *                 (needs cta_group 0 or 1 and one consumer): single CTAs
 *                 with 128 x 64 tiles and an 8-stage ring (all of a K up to
 *                 512 in flight after one load latency), D stored by
 *                 coalesced warp stores; for small, latency-bound problems.
 *                 16 (needs cta_group 0 or 1, one consumer, block_m 0 or 64,
 *                 cluster_k 0 or 1): thin single-CTA 64 x 16 tiles, MMAs of
 *                 M = 64, N = 16, 32 columns of tensor memory, a ring of 3
 *                 stages of four K tiles, each row of D stored straight from
 *                 registers; for the shortest problems.
 *                 Not on the pages: they fix the tile at 128 or 256 x 256.  0
 *                 (default): 64 when cta_group is 0, consumers is not 2 and
 *                 the 128 x 64 tiles fit one wave of co-resident CTAs (with
 *                 a workspace, unless no cluster K split applies and split-K
 *                 over 256-wide tiles would take 8 slices or more), else
 *                 256; and with block_m
 *                 and cluster_k at 0 too, 16 where the tiny tiles of block_m
 *                 64 would run a K-loop of at most 12 tiles of 64 and the
 *                 64 x 16 tiles fill at most half of the co-resident CTAs.
 *                 Other values:
 *                 GEMM_ERR_INVALID_ARG.
 *   block_m       rows of D per CTA.  128: the tiles above.  64 (needs
 *                 block_n 0 or 64, which then means 64): single CTAs with
 *                 64 x 64 tiles, MMAs of M = 64 and a ring of 6 stages of
 *                 two K tiles each; for the
 *                 smallest problems.  Not on the pages.  0 (default): with
 *                 block_n resolved to 64, 64 when the 64 x 64 tiles number at
 *                 most two thirds of the co-resident CTAs, else 128.  Other
 *                 values:
 *                 GEMM_ERR_INVALID_ARG.
 *   cluster_k     2, 4 or 8 (needs block_n 0 or 64, which then means 64, and
 *                 one single-CTA consumer; block_m 0 then means 64): tiny
 *                 (block_m 64) or narrow (block_m 128) tiles with K split
 *                 across a thread-block cluster of that many CTAs, one
 *                 cluster per tile and one K slice per CTA (at most one per
 *                 64-wide K tile, so fewer CTAs when K is short, and halved
 *                 until the device can run clusters of that size).  Each CTA
 *                 keeps its slice's fp32 sums in shared memory and the
 *                 cluster adds them, in slice order, through distributed
 *                 shared memory before the one rounding to fp16: no
 *                 workspace and no second kernel.  Each CTA then streams
 *                 1/cluster_k of the tile's operands, which is what bounds
 *                 small problems.  Not on the pages.  1: no K split.
 *                 0 (default): with max_clusters 0 and at least 8 K tiles
 *                 of 64 (12 for tiny tiles), the largest of 8, 4, 2 that
 *                 leaves each CTA at least 2 K tiles, lets all the clusters
 *                 run at once and keeps the grid within half the co-resident
 *                 CTAs (a quarter for tiny tiles in clusters of 8; within
 *                 all of them from 24 K tiles per CTA), else 1.  With
 *                 block_m 0 as well, a long K can turn tiny tiles into
 *                 narrow ones: where the tiny tiles get no split but the
 *                 narrow ones do with at least 16 K tiles per CTA, and where
 *                 the tiny ones split in 2 but the narrow ones can split in
 *                 4 with at least 8.  max_clusters does not cap this grid.
 *                 Other values: GEMM_ERR_INVALID_ARG.
 */
typedef struct gemm_f16_options {
    int32_t cta_group;
    int32_t max_clusters;
    int32_t raster_group;
    int32_t debug_flags;
    int64_t timeout_ns;
    int32_t overlap_launch;
    int32_t consumers;
    int32_t block_n;
    int32_t block_m;
    int32_t cluster_k;
} gemm_f16_options;

/*
 * 1 if gemm_f16_nt() accepts this shape, 0 if not.  Pure host logic, no CUDA
 * call.  Accepted: M >= 0, N >= 0, K >= 0, N % 8 == 0 and K % 8 == 0 (rows of
 * B and D are then whole 16-byte units, as the tensor-memory-accelerator copy
 * engine requires), and M, N, K <= 2^31 - 1024 (tile coordinates are 32-bit
 * integers; the margin keeps a last tile's rows and columns from wrapping).
 * M, N and K need not be multiples of
 * the tile: edge tiles read zeros past the ends of A and B and write only the
 * in-range part of D.  M == 0 or N == 0 is an empty product (nothing is
 * launched); K == 0 writes D = 0.
 */
int gemm_f16_nt_supported(int64_t M, int64_t N, int64_t K);

/*
 * D = A * B^T (see the top of this file) with the default options.
 * Returns GEMM_OK once the kernel is enqueued on `stream`; GEMM_ERR_INVALID_ARG
 * for a null A/B/D with a non-empty product or negative sizes;
 * GEMM_ERR_UNSUPPORTED_SHAPE; GEMM_ERR_MISALIGNED; GEMM_ERR_NO_DEVICE;
 * GEMM_ERR_ARCH; GEMM_ERR_LAUNCH.
 */
int gemm_f16_nt(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *stream);

/* As gemm_f16_nt(), with options (NULL = defaults); GEMM_ERR_INVALID_ARG for
 * an option out of range. */
int gemm_f16_nt_ex(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *stream,
                   const gemm_f16_options *opts);

/*
 * End to end from host memory: enqueues on `stream`, in order, the copies of the
 * host operands A_host (M x K) and B_host (N x K) into the caller's device
 * buffers A_dev and B_dev, the GEMM D_dev = A_dev * B_dev^T of gemm_f16_nt_ex()
 * with `opts` (NULL = defaults), and the copy of D_dev into the host buffer
 * D_host (M x N); returns once all four are enqueued.  D_host is complete when
 * the stream reaches that point (synchronise the stream, or an event recorded
 * after the call, before reading it).  Layouts as above, all fp16 row-major.
 * The device buffers are owned by the caller and the library allocates
 * nothing: D_dev must not overlap A_dev or B_dev; they must stay alive, and
 * not be written by other work, until the stream has passed the copy-out.
 * With page-locked (pinned) host buffers the copies are asynchronous and
 * overlap work on other streams: calls on two or three streams, each with its
 * own device buffers, overlap one step's copy-in, another's GEMM and a third's
 * copy-out, which is how a stream of host-resident problems is best run.
 * With pageable host buffers the copy-in returns only when the host data has
 * been taken.  Errors: those of gemm_f16_nt_ex() for the device buffers (all
 * checked before anything is enqueued), GEMM_ERR_INVALID_ARG for a null host
 * buffer of a non-empty product, GEMM_ERR_CUDA when a copy cannot be
 * enqueued.  Not on the pages, which start from operands in device memory.
 */
int gemm_f16_nt_host(const void *A_host, const void *B_host, void *D_host, int64_t M, int64_t N, int64_t K,
                     void *A_dev, void *B_dev, void *D_dev, void *stream, const gemm_f16_options *opts);

/*
 * As gemm_f16_nt_ex(), with a caller-owned device workspace that lets the
 * library split the K-loop across CTA pairs when the output has few tiles
 * (split-K: at most a quarter as many 256x256 tiles as co-resident pairs, and
 * at least 32 K tiles of 64; the pages' persistent scheduler, TIRx notes V6,
 * would otherwise leave most SMs idle for the whole K-loop).  With the default
 * options a problem whose narrow 128 x 64 tiles fit one wave (see block_n)
 * takes those instead, unless the split would cut K into at least 8 slices;
 * and a problem whose narrow or tiny tiles split K across a cluster
 * (cluster_k) takes that, which needs no workspace and is faster, so with
 * the defaults this workspace serves mostly grids capped by max_clusters and
 * calls that ask for 256-wide tiles.
 * K is then cut into S slices (4..16); each slice's fp32 partial sums go to the workspace
 * as [S][M][N] fp32 and a second kernel on `stream` adds them in fp32 and
 * rounds once to fp16.  `workspace` is a device pointer, 16-byte aligned,
 * owned by the caller, needing no initialisation; its contents are scratch
 * (overwritten by each call, meaningless afterwards) and it must not be used
 * by two calls that may overlap on the GPU.  If workspace_bytes is smaller
 * than gemm_f16_nt_workspace_size() for the same arguments, or the pointer is
 * misaligned, the call runs without split-K.  NULL with 0 bytes is allowed
 * (= gemm_f16_nt_ex).  Errors as gemm_f16_nt_ex(), and GEMM_ERR_INVALID_ARG for
 * a NULL workspace with a non-zero size or a negative size.
 */
int gemm_f16_nt_ws(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *workspace,
                   int64_t workspace_bytes, void *stream, const gemm_f16_options *opts);

/*
 * Bytes of workspace gemm_f16_nt_ws() will use for these arguments on the
 * current device (S * M * N * 4 with split-K, 0 when it would not split), or
 * a negative gemm_status_t (bad options or shape, no usable device).  The
 * choice depends on how many clusters fit on the device, so this makes the
 * same per-device set-up as the first GEMM call (no GPU work is enqueued).
 */
int64_t gemm_f16_nt_workspace_size(int64_t M, int64_t N, int64_t K, const gemm_f16_options *opts);

/*
 * Bytes of the library's fixed device scratch array used by
 * gemm_f16_nt_static_ws().
 */
#define GEMM_F16_STATIC_SCRATCH_BYTES (16ll << 20)

/*
 * As gemm_f16_nt_ws(), but the split-K scratch is a fixed array inside this
 * library (GEMM_F16_STATIC_SCRATCH_BYTES = 16 MiB per GPU) instead of memory
 * the caller passes, so the call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.  It is for callers that cannot
 * allocate device memory while they run -- code that fixes its memory budget
 * once and forbids later allocation, a plug-in inside an application that
 * owns the GPU's memory, or a loop where an allocation (which may block and
 * synchronise the device) is not allowed.  The pages have no counterpart of
 * this entry point; it is a property of this library, not of the method.
 *
 * A, B, D, M, N, K, stream and opts mean what they mean for gemm_f16_nt_ex().
 * The first call on each device also resolves the array's device address (and
 * does the per-device set-up every first call does); make that first call
 * before any stream capture.  Every GPU that loads this library's device code
 * holds the array until the process exits.  All calls on a device share it
 * and it keeps the last call's contents; nothing in it needs to start at
 * zero, but calls that may overlap on the GPU race on it, so order them (one
 * stream, or events).  Returns GEMM_ERR_SCRATCH_LIMIT, before anything is
 * enqueued, when the split-K scratch the problem would use
 * (gemm_f16_nt_workspace_size()) exceeds the array; otherwise the errors of
 * gemm_f16_nt_ex().
 */
int gemm_f16_nt_static_ws(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K, void *stream,
                          const gemm_f16_options *opts);

/* What a call would launch (see gemm_f16_nt_describe()). */
typedef struct gemm_f16_launch_info {
    int32_t cta_group;        /* 1 or 2 */
    int32_t consumers;        /* 1 or 2 */
    int32_t block_n;          /* tile width: 256, 64 or 16 */
    int32_t split_k;          /* K slices S (1 = no split-K; > 1 adds the reduction kernel) */
    int32_t block_m;          /* rows of D per CTA and consumer: 128 or 64 */
    int32_t stages;           /* K tiles of 64 the shared-memory operand ring holds (tiny tiles
                                 move two per ring slot, thin tiles four) */
    int64_t clusters;         /* clusters in the grid (CTAs = clusters * cta_group * cluster_k); persistent
                                 unless cluster_k > 1, which runs one cluster per tile */
    int64_t work_items;       /* tiles, half tiles or K slices dealt to the clusters (to the CTAs with
                                 cluster_k > 1) */
    int64_t workspace_bytes;  /* split-K partials, 0 without split-K */
    int32_t cluster_k;        /* CTAs sharing one tile's K (1 = none; see gemm_f16_options) */
} gemm_f16_launch_info;

/*
 * The configuration gemm_f16_nt_ex() (with_workspace 0) or gemm_f16_nt_ws()
 * with a large enough workspace (with_workspace 1) would launch for these
 * arguments on the current device, without launching anything: the choices
 * described under gemm_f16_options, resolved.  Makes the same per-device
 * set-up as the first GEMM call.  Not on the pages.  Returns GEMM_OK and
 * fills *out (all zero when M, N or K is 0: then nothing, or only a fill of D
 * with zeros, is launched), or the errors of gemm_f16_nt_workspace_size(),
 * and GEMM_ERR_INVALID_ARG for a null `out` or with_workspace not 0 or 1.
 */
int gemm_f16_nt_describe(int64_t M, int64_t N, int64_t K, const gemm_f16_options *opts, int32_t with_workspace,
                         gemm_f16_launch_info *out);

/*
 * Kernel configurations whose co-resident cluster counts steer the choices of
 * gemm_f16_options (see gemm_f16_co_resident()).
 */
#define GEMM_F16_CONFIG_KINDS 11

/*
 * How many clusters of each kernel configuration fit on the current device at
 * once (cudaOccupancyMaxActiveClusters, measured at the per-device set-up the
 * first GEMM call makes), in this order: [0] single CTAs with 128 x 256 tiles,
 * [1] CTA pairs, [2] CTA pairs with two consumers, [3] narrow 128 x 64 tiles,
 * [4] tiny 64 x 64 tiles, [5] [6] [7] tiny tiles with K split across clusters
 * of 2, 4 and 8 CTAs, [8] [9] [10] narrow tiles likewise (0: the device cannot
 * run that split).  `count` must be GEMM_F16_CONFIG_KINDS.  Returns GEMM_OK, the
 * errors of the device set-up, or GEMM_ERR_INVALID_ARG.  Not on the pages.
 */
int gemm_f16_co_resident(int32_t *out, int32_t count);

/*
 * As gemm_f16_nt_describe(), for a device with the given co-resident counts
 * (the order of gemm_f16_co_resident(); the first five at least 1, the rest
 * at least 0) instead of the current one: pure host logic, no CUDA call.  On
 * the current device, with its own counts, it gives what
 * gemm_f16_nt_describe() gives.  Errors as gemm_f16_nt_describe(), and
 * GEMM_ERR_INVALID_ARG for a null or short `co_resident`.  Not on the pages.
 */
int gemm_f16_nt_describe_for(int64_t M, int64_t N, int64_t K, const gemm_f16_options *opts, int32_t with_workspace,
                             const int32_t *co_resident, int32_t count, gemm_f16_launch_info *out);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: GEMM_OK, or GEMM_ERR_DEVICE_TIMEOUT if a wait inside a kernel ran out
 * (the kernel then skipped its remaining work and exited; D is incomplete),
 * or, from the checked build of the library (compiled with
 * -DGEMM_F16_DEVICE_CHECKS=1 for tests), GEMM_ERR_DEVICE_BOUNDS if a range
 * check inside a kernel failed.  If `info` is not NULL it receives where the
 * first failure happened: bits 56-63 role (1 producer, 2 MMA issuer, 3
 * epilogue), 0-31 the tile's sequence number in that CTA, and 32-55 the CTA
 * index for a timeout, or 48-55 the check (1 work item, 2 ring stage, 3 TMEM
 * columns, 4 epilogue chunk, 5 staging buffer, 6 the rows a CTA adds up in a
 * K split across a cluster) and 32-47 the CTA index for a
 * failed range check.  Returns GEMM_ERR_CUDA if the
 * synchronisation itself reports an error.
 */
int gemm_f16_last_device_status(void *stream, uint64_t *info);

/* A static, human-readable name for a gemm_status_t value. */
const char *gemm_f16_status_string(int status);

/* One unit of work of a persistent cluster (see gemm_f16_nt_schedule()). */
typedef struct gemm_f16_work_item {
    int64_t m_idx, n_idx;     /* the tile: rows m_idx * block_m*cta_group*consumers, columns n_idx * block_n */
    int64_t n_off, n_len;     /* columns n_off .. n_off + n_len of that tile (block_n, or a half) */
    int64_t slice;            /* K slice under split-K, else 0 */
    int64_t kt_begin, kt_end; /* 64-wide K tiles [kt_begin, kt_end) */
} gemm_f16_work_item;

/*
 * The persistent scheduler, as a pure host query (no CUDA call); the kernel
 * runs the same code.  D is cut into tiles of (block_m * cta_group *
 * consumers) rows x block_n columns (consumers 0 means 1; block_m 0 means 64
 * with block_n 16, else 128, and 64, the tiny tiles of gemm_f16_options, needs
 * block_n 0, 16 or 64; block_n 0 means 64 with block_m 64, else 256; block_n
 * 64 or 16, the narrow and thin tiles, needs cta_group 0 or 1, which then
 * means 1, and one consumer, and 16 needs block_m 64), ordered in groups of
 * `raster_group` M-tiles (0 = the shape-derived default described under
 * gemm_f16_options): M fastest inside a group, then N, then the next group
 * (TIRx notes V6, "Better L2 Locality").  With T tiles and P = num_clusters
 * persistent clusters, if the last wave is at most half full (T = qP + r,
 * 0 < 2r <= P) its r tiles are split along N into 2r half tiles of 128
 * columns, so that the tail lasts half a tile (V6 notes that 1024 tiles over
 * 148 CTAs leave 6.9 tiles per CTA, i.e. a partly idle last wave).  With
 * split_k = 1 (what gemm_f16_nt_ws() does given enough workspace) and few
 * tiles, K is instead cut into slices: item t*S + s is slice s of tile t.
 * Narrow, tiny and thin tiles are never split along N, nor along K this way.
 * split_k 2, 4 or 8 (narrow or tiny tiles) is the K split across a cluster
 * (cluster_k of gemm_f16_options): S = split_k, reduced to at most the
 * number of 64-wide K tiles, with the same item numbering; that kernel runs
 * one item per CTA, so pass num_clusters = T * S and iter 0 (CTA i of the
 * grid runs item i; the S CTAs of tile t form one cluster).
 * Cluster `cluster_id` takes work items cluster_id, cluster_id + P, ...
 * Returns 1 and fills *out with the iter-th item of that cluster, 0 if the
 * cluster has no iter-th item, or GEMM_ERR_INVALID_ARG for bad arguments.
 */
int gemm_f16_nt_schedule(int64_t M, int64_t N, int64_t K, int32_t cta_group, int32_t consumers, int32_t block_n,
                         int32_t block_m, int32_t raster_group, int32_t split_k, int64_t num_clusters,
                         int64_t cluster_id, int64_t iter, gemm_f16_work_item *out);

/*
 * Where CTA `rank` of a work item reads and writes, as a pure host query (no
 * CUDA call); the kernel uses the same function.  TIRx notes V8, "Operand
 * Partition" and "Output Ownership": with bm = block_m (0 meaning 64 with
 * block_n 16, else 128), m_base =
 * m_idx * bm * cta_group * consumers and n_base = n_idx * block_n + n_off, the
 * CTA loads A rows a_row = m_base + bm * rank (bm rows; consumer c's block
 * lies c * bm * cta_group rows further, TIRx notes V9) and B rows b_row =
 * n_base + (n_len / cta_group) * rank (n_len / cta_group rows, shared by the
 * consumers), and writes D rows d_row = a_row (bm rows per consumer) over the
 * n_len columns starting at d_col = n_base ("Epilogue Column Address": no rank
 * term).  block_n is 0 (meaning 256, or 64 with block_m 64) or 256: n_len is
 * 256 (whole tile, n_off 0) or 128 (half tile, n_off 0 or 128); or 64 (narrow
 * tiles, cta_group 0 or 1, one consumer): n_len 64, n_off 0; or 16 (thin
 * tiles, also block_m 64): n_len 16, n_off 0.  block_m 64 needs block_n 0, 16
 * or 64.  Returns GEMM_OK, or GEMM_ERR_INVALID_ARG (cta_group not
 * 0/1/2, consumers not 0/1/2 or 2 without a pair, block_n not 0/16/64/256 or
 * 16 or 64 with a pair or two consumers, block_m not 0/64/128, 64 with
 * block_n 256 or 128 with block_n 16,
 * rank out of range, bad n_off/n_len, negative or too large indices, null
 * outputs).
 */
int gemm_f16_nt_cta_origin(int32_t cta_group, int32_t consumers, int32_t block_n, int32_t block_m, int64_t m_idx,
                           int64_t n_idx, int64_t n_off, int64_t n_len, int32_t rank, int64_t *a_row, int64_t *b_row,
                           int64_t *d_row, int64_t *d_col);

/*
 * The stage/phase bookkeeping of one SMEM or TMEM ring, run on the host with
 * the same code the kernel runs ("GEMM III", "Four barriers = two
 * producer-consumer rings": PipelineState(depth, phase) with .stage, .phase
 * and .advance(); TIRx notes V5 "Barrier Phase Tracking").  Writes the
 * (stage, phase) seen before each of `steps` advances.  Returns GEMM_OK, or
 * GEMM_ERR_INVALID_ARG (depth outside 1..16, phase not 0/1, null outputs).
 */
int gemm_f16_pipeline_trace(int32_t depth, int32_t initial_phase, int32_t steps, int32_t *stage_out,
                            int32_t *phase_out);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H */
