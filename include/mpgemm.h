/*
 * mpgemm: mixed-precision GEMM for one NVIDIA GB300 (sm_103a).
 *
 *     C = alpha * A * B + beta * C
 *
 * A is M x K and B is K x N, both row-major IEEE binary16 (FP16). C is M x N,
 * row-major IEEE binary32 (FP32). Products are accumulated in FP32 on the
 * fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
 *
 * The operation is the one defined on "Day 80, Capstone 4: a tensor-core
 * GEMM" (sections "Capability" and "Minimal model": FP16 inputs, FP32
 * accumulation and FP32 C, correct when no tile divides the matrix), with
 * the alpha/beta scaling of the matched cublasGemmEx baseline that page and
 * "Day 72: Tensor cores with WMMA" ("Why this program calls cuBLAS twice")
 * compare against. The pages' own gate entry point ("Independent gate":
 * solve(a, b, c, m, n, k, stream)) takes no alpha, beta or leading
 * dimensions; this interface adds them in the BLAS way.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Element (i, k) of A is A[i*lda + k]; (k, j) of B is B[k*ldb + j];
 *    (i, j) of C is C[i*ldc + j]. lda >= max(1, K), ldb >= max(1, N),
 *    ldc >= max(1, N). Any leading dimension is accepted. When A's rows do
 *    not start on 16-byte boundaries (an odd lda, say) and B is row-major,
 *    the tensor-core pass reads A directly in classes of rows that share a
 *    misalignment (their offset modulo 16 bytes, or, in the 256 x 288 and
 *    256 x 320 CTA-pair tiles, their offset in a 128-byte line); otherwise
 *    an operand whose base address or row pitch is not a multiple of 16
 *    bytes is staged through an aligned copy on the device first. A class
 *    is read from the aligned address at or below its first row, up to 126
 *    bytes before A: A's allocation must begin on a 128-byte boundary, as
 *    every CUDA device allocation does (those bytes are read, never used).
 *  - A and B must be aligned to 2 bytes and C to 4 bytes (their element
 *    sizes); otherwise MPGEMM_ERR_INVALID_VALUE.
 *  - beta == 0: C is only written, never read, so it may hold NaN on entry.
 *    alpha == 0 or K == 0: A and B are not read and C = beta * C.
 *    M == 0 or N == 0: nothing happens.
 *  - Every dimension must be below 2^31, and M*N*K below 2^62.
 *  - `stream` is a cudaStream_t (or CUstream) passed as void*; NULL is the
 *    legacy default stream. Device entry points are asynchronous: they
 *    enqueue work on `stream` and return without synchronising. The GEMM
 *    kernel is launched with programmatic stream serialization: its CTAs may
 *    be scheduled and set up (barriers, tensor memory) while the previous
 *    kernel of the stream finishes, but they read and write no global memory
 *    before that kernel has completed, so stream order holds as usual.
 *  - The caller owns A, B, C and the stream. The handle owns its workspace
 *    (aligned staging copies, grown on demand with stream-ordered
 *    allocation), the tensor-core launch configuration and a status word
 *    that the device writes if one of its bounded waits gives up.
 *  - A handle is bound to the device that was current at mpgemm_create:
 *    calls through it return MPGEMM_ERR_INVALID_VALUE (and enqueue nothing)
 *    while another device is current. It may be used from one stream at a
 *    time (its workspace is reused in stream order); use one handle per
 *    concurrently used stream. A handle is not thread-safe: two host threads
 *    must not call it at the same time. Any host thread may call it.
 */
#ifndef MPGEMM_H
#define MPGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mpgemm_handle_st* mpgemm_handle_t;

typedef enum {
    MPGEMM_OK = 0,
    MPGEMM_ERR_INVALID_VALUE = 1,      /* bad argument; nothing was enqueued */
    MPGEMM_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
    MPGEMM_ERR_ALLOC = 3,              /* device or pinned host allocation failed */
    MPGEMM_ERR_LAUNCH = 4,             /* a kernel launch or copy could not be enqueued */
    MPGEMM_ERR_DEVICE_TIMEOUT = 5,     /* a device wait gave up (reported by a later call) */
    MPGEMM_ERR_CUDA = 6,               /* another CUDA runtime or driver error */
    MPGEMM_ERR_SCRATCH_LIMIT = 7       /* mpgemm_run_noalloc: the operands need more staging
                                          scratch than its fixed area holds; nothing enqueued */
} mpgemm_status_t;

/* Create a handle bound to the current CUDA device. Fails with
 * MPGEMM_ERR_UNSUPPORTED_DEVICE unless that device is compute capability
 * 10.3 (GB300). *out is set to NULL on failure. (No page defines this call:
 * the pages' gate entry point takes no handle. The handle holds the
 * stream-ordered workspace, the encoded tensor maps and the device status
 * word.) */
mpgemm_status_t mpgemm_create(mpgemm_handle_t* out);

/* Release the handle and its workspace. NULL is accepted. Work enqueued
 * with the handle must have completed (synchronise its stream first). (No
 * page defines this call: it ends the lifetime mpgemm_create starts.) */
mpgemm_status_t mpgemm_destroy(mpgemm_handle_t h);

/* C = alpha*A*B + beta*C on device memory (see the conventions above).
 * A, B and C are device pointers. Invalid arguments return
 * MPGEMM_ERR_INVALID_VALUE before anything is enqueued. If an earlier call
 * on this handle reported a device timeout that was not yet collected,
 * this call returns MPGEMM_ERR_DEVICE_TIMEOUT without enqueuing work and
 * clears the report. */
mpgemm_status_t mpgemm_run(mpgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                           float alpha, const void* A, int64_t lda,
                           const void* B, int64_t ldb,
                           float beta, float* C, int64_t ldc, void* stream);

/* Layout of B for mpgemm_run_ex. */
typedef enum {
    MPGEMM_B_ROW_MAJOR = 0,   /* (k, j) at B[k*ldb + j], ldb >= max(1, N) (as mpgemm_run) */
    MPGEMM_B_COL_MAJOR = 1    /* (k, j) at B[j*ldb + k], ldb >= max(1, K): B stored as N rows
                                 of K, the layout of the capstone gate's solve() */
} mpgemm_b_layout_t;

/* mpgemm_run with a choice of B layout; everything else as mpgemm_run. */
mpgemm_status_t mpgemm_run_ex(mpgemm_handle_t h, mpgemm_b_layout_t b_layout,
                              int64_t M, int64_t N, int64_t K,
                              float alpha, const void* A, int64_t lda,
                              const void* B, int64_t ldb,
                              float beta, float* C, int64_t ldc, void* stream);

/* The interface of "Day 80, Capstone 4: a tensor-core GEMM", section
 * "Independent gate": C = A * B with A (m x k) row-major, B (k x n)
 * column-major and C (m x n) row-major, all densely packed (lda = k,
 * ldb = k, ldc = n), asynchronous on `stream`. The first call on a device
 * creates a handle for that device that lives until the process exits (if
 * that creation fails, its status is returned and the next call on the
 * device tries again); all
 * calls on a device share its workspace, so calls on different streams of
 * one device must not overlap on the GPU (use mpgemm_run_ex with a handle
 * per stream for that). Host threads may call it concurrently: the calls
 * on one device are serialised on the host while they are enqueued. */
mpgemm_status_t mpgemm_solve(const void* a, const void* b, float* c,
                             size_t m, size_t n, size_t k, void* stream);

/* The same operation on HOST buffers: A, B (and C when beta != 0) are
 * copied to device workspace owned by the handle, the GEMM runs there and
 * C is copied back, all in order on `stream`. Host buffers may be pageable
 * or pinned (pinned buffers make the copies asynchronous). The caller must
 * synchronise `stream` before reading C or releasing the host buffers. */
mpgemm_status_t mpgemm_run_host(mpgemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                float alpha, const void* A, int64_t lda,
                                const void* B, int64_t ldb,
                                float beta, float* C, int64_t ldc, void* stream);

/* Synchronise `stream`, then report the state of the handle's device status
 * word (no page defines this call: it reports the bounded device waits this
 * library adds): MPGEMM_OK, or MPGEMM_ERR_DEVICE_TIMEOUT if a bounded device wait gave
 * up since the last report (the report is cleared), or MPGEMM_ERR_CUDA if
 * the synchronisation itself failed. If info is not NULL it receives four
 * integers describing the last timeout: {code, role, block, detail}
 * (all zero when there was none). */
mpgemm_status_t mpgemm_sync_status(mpgemm_handle_t h, void* stream, int32_t info[4]);

/* Tunables and test switches, set per handle. */
typedef enum {
    MPGEMM_OPT_TILE_N = 1,        /* 0 = automatic (default), or columns per tile: 128 or 256
                                     (one CTA, or a pair with TILE_M 256); 320 (one CTA per
                                     128 x 320 tile, or with TILE_M 256 a pair per 256 x 320
                                     tile, row-major B only); 288, 384 and 512 (a cluster of
                                     two CTAs per 256-row tile; 288 with row-major B only).
                                     A combination not listed makes runs return
                                     INVALID_VALUE. Automatically, N from 257 to 288, 320 or
                                     384 in one column of 288-, 320- or 384-wide pairs when
                                     those fill every pair */
    MPGEMM_OPT_MAX_CTAS = 2,      /* 0 = one persistent CTA per SM (default), else an upper bound */
    MPGEMM_OPT_FORCE_STAGING = 3, /* 1 = stage A and B through aligned copies even when aligned */
    MPGEMM_OPT_WAIT_LIMIT_US = 4, /* limit of every bounded device wait, microseconds (default 4e6) */
    MPGEMM_OPT_RASTER_GROUP = 5,  /* M-tiles per rasterisation group, 0 = automatic (default) */
    MPGEMM_OPT_TEST_STALL = 6,    /* test only: 1 = the load warp issues no loads, so the
                                     kernel's bounded waits expire and a timeout is reported */
    MPGEMM_OPT_TILE_M = 7,        /* 0 = automatic (default); 128 = one CTA per tile;
                                     256 = a cluster of two CTAs per 256 x 256 tile
                                     (256 x 512 when TILE_N is 512). TILE_M 128 with
                                     TILE_N 512 makes runs return INVALID_VALUE */
    MPGEMM_OPT_L2_KEEP = 8,       /* L2 hints for the operand loads: 0 = automatic (default:
                                     both evict-last, except an operand that only one tile
                                     reads, i.e. A when N fits one tile column or B when M
                                     fits one row block, which is evict-first),
                                     1 = keep A (B evict-first), 2 = keep B (A evict-first) */
    MPGEMM_OPT_SPLIT_K = 9,       /* 0 = automatic (default): when the one-CTA output tiles
                                     occupy at most a quarter of the SMs and K has 32 or more
                                     64-wide blocks (half of the SMs and 16 blocks when
                                     beta == 1), or at most an eighth of the SMs and K has 8
                                     or more blocks (up to five slices), each
                                     tile's K range is cut into slices whose
                                     partial products are summed: in clusters (see
                                     SPLIT_REDUCE) or added into C after C = beta*C;
                                     1 = never; n in 2..64 = n slices (one-CTA tiles only) */
    MPGEMM_OPT_C_STORE = 10,      /* 0 = automatic (default): C is written with tiled TMA stores
                                     when beta == 0 and K is not split, or added to with tiled
                                     TMA reduce-adds when K is split (C then holds beta*C
                                     first), provided A is read as one row class, C's base and
                                     ldc are 16-byte aligned and N is a multiple of 4; 1 = always
                                     one store (or atomic add) per lane (the path used in every
                                     other case) */
    MPGEMM_OPT_ACCUMULATOR = 11,  /* 0 or 32 = FP32 accumulators (default, the operation defined
                                     above); 16 = FP16 accumulators, a study variant of "Day 72:
                                     Tensor cores with WMMA" (Exercise: AccT = __half): every
                                     K = 16 step is rounded to FP16, so sums lose low bits once
                                     they pass 2048 and overflow to infinity past 65504 ("Day 80,
                                     Capstone 4", "Common failures"). K is never split then: the
                                     whole K range accumulates in one FP16 accumulator. Not for
                                     production use. */
    MPGEMM_OPT_REPRODUCIBLE = 12, /* 0 = default: a call may split K (see SPLIT_K), and slices
                                     that add into C do so in the order they arrive, so
                                     results may differ in the last bits between identical
                                     calls (always within the stated tolerance; exact inputs
                                     stay exact); 1 = K is split only where the slices are
                                     summed in clusters (SPLIT_REDUCE), in a fixed order, so
                                     identical calls give identical bits (every tile shape sums in a fixed
                                     order: the two MMA threads of a 256 x 512 CTA-pair tile
                                     own disjoint columns of the accumulator, and those of a
                                     256 x 256 tile hand alternate k-blocks to each other
                                     strictly in turn). The stream-K walk (STREAM_K) is
                                     allowed: it, too, sums in a fixed order. */
    MPGEMM_OPT_STREAM_K = 13,     /* 0 = automatic (default): CTA-pair tiles of 288, 320 or 384
                                     columns (N from 257 to 384), or a single column of
                                     256-wide pair tiles, that leave the last wave of
                                     pairs partly idle walk the problem as one contiguous range
                                     of k-blocks per pair instead of whole tiles (stream-K,
                                     Osama et al., 2023): every pair gets the same number of
                                     k-blocks, and a tile cut between two ranges is written
                                     twice in a fixed order (the later k-blocks with beta * C
                                     first, then the earlier ones added on), so identical calls
                                     still give identical bits; 1 = never; 2 = whenever the
                                     call runs on CTA pairs of 256 to 384 columns with at least
                                     one tile per pair (not with FP16 accumulators, nor in
                                     mpgemm_run_noalloc) */
    MPGEMM_OPT_SPLIT_REDUCE = 14  /* how split-K slices are summed. 1 = they add into C with
                                     TMA reduce-adds or atomic adds, after a pass that applies
                                     beta (unless beta == 1), in the order they finish.
                                     2 = in clusters, where the tiles are 128 x 128 with at
                                     most 8 slices (more are cut to 8) and every slice fits
                                     the device at once: the slices of a tile run as one
                                     cluster of CTAs; each writes its partial accumulator to
                                     its shared memory and, after a cluster barrier, sums its
                                     share of the tile's rows over the partials (through
                                     distributed shared memory, in CTA order) and writes C
                                     once, with no pass over C first and no atomics, so
                                     identical calls give identical bits; else as 1. About
                                     1.3-4 us slower per call than 1 on GB300.
                                     0 = automatic (default): 2 when REPRODUCIBLE is set, else 1 */
} mpgemm_option_t;

/* Set an option. Unknown options or out-of-range values return
 * MPGEMM_ERR_INVALID_VALUE and leave the handle unchanged. */
mpgemm_status_t mpgemm_set_option(mpgemm_handle_t h, mpgemm_option_t opt, int64_t value);

/* What mpgemm_run_ex would do for these arguments with this handle's options
 * and device (host work only; the handle's device must be current). Same
 * argument checks and status codes as mpgemm_run_ex. */
typedef struct mpgemm_plan_s mpgemm_plan_t;
mpgemm_status_t mpgemm_plan_call(mpgemm_handle_t h, mpgemm_b_layout_t b_layout, int64_t M, int64_t N,
                                 int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                                 int64_t ldb, float beta, const float* C, int64_t ldc, mpgemm_plan_t* out);

/* What mpgemm_run would do for these arguments, computed on the host only
 * (no device work; usable without a GPU). `num_sms` stands in for the
 * device's SM count; tile_m, tile_n, max_ctas and force_staging mirror the
 * options above; b_col_major selects the layout of B (ldb >= K when set). The grid of the CTA-pair kernel is further capped at run
 * time by the number of two-CTA clusters the device can hold at once. */
struct mpgemm_plan_s {
    int32_t quick;          /* 0 = tensor-core path, 1 = nothing to do, 2 = C = beta*C only */
    int32_t stage_a;        /* 1 if A is copied to an aligned buffer first */
    int32_t stage_b;        /* 1 if B is copied to an aligned buffer first */
    int32_t tile_m;         /* rows per output tile: 128 (one CTA) or 256 (a CTA pair) */
    int32_t tile_n;         /* columns per output tile (128, 256 or 320; 256, 288, 320, 384 or
                               512 for a pair) */
    int32_t tile_k;         /* K per pipeline stage (64, or 128 for tiles that stage two
                               64-wide k-blocks at once); k_blocks counts these stages */
    int32_t stages;         /* shared-memory pipeline depth */
    int32_t m_tiles, n_tiles, k_blocks;
    int64_t tiles;          /* m_tiles * n_tiles */
    int32_t grid;           /* persistent CTAs launched */
    int32_t raster_group;   /* M-tiles walked per column band */
    int32_t smem_bytes;     /* dynamic shared memory per CTA */
    int32_t last_k_valid;   /* valid K columns in the last pipeline stage */
    int64_t workspace_bytes;/* device staging bytes the call needs */
    int32_t split_tiles;    /* tiles of the last partial wave done as two half-width items */
    int64_t items;          /* work items the persistent CTAs walk: tiles + split_tiles, or
                               tiles * k_splits */
    int32_t k_splits;       /* slices of K per tile (1 = no split-K) */
    int32_t a_classes;      /* 0: A is read through one plain tensor map (aligned, or staged);
                               P >= 1: A's rows are not 16-byte aligned and are read in P
                               classes of rows i = r (mod P) instead of being copied: rows
                               at the same offset modulo 16 bytes (P <= 8), or, in the
                               256 x 288 and 256 x 320 pairs when that adds at most 1/32
                               more tiles, in the same 128-byte line (P <= 64) */
    int32_t sk_ranges;      /* 0, or the stream-K walk's ranges of k-blocks (one per CTA pair;
                               see MPGEMM_OPT_STREAM_K) */
    int32_t split_reduce;   /* k_splits > 1: 1 = a tile's slices run as one cluster and are
                               summed through distributed shared memory; 0 = they add into C
                               (see MPGEMM_OPT_SPLIT_REDUCE) */
};

mpgemm_status_t mpgemm_plan(int64_t M, int64_t N, int64_t K, float alpha,
                            const void* A, int64_t lda, const void* B, int64_t ldb,
                            float beta, const float* C, int64_t ldc,
                            int32_t num_sms, int32_t tile_m, int32_t tile_n, int32_t max_ctas,
                            int32_t force_staging, int32_t b_col_major, mpgemm_plan_t* out);

/* C = alpha*A*B + beta*C on device memory, like mpgemm_run, for callers that
 * cannot allocate: no handle, and no device or host allocation of any kind
 * (no cudaMalloc, cudaMallocAsync, cudaHostAlloc or allocating library call)
 * at any call. Such callers include code that runs where the allocator must
 * not be touched (inside another library's fixed memory-pool budget, or on
 * a path that runs when device memory is already exhausted, where a new
 * allocation would fail), and code that cannot own a handle's lifetime. The pages have no counterpart of this
 * entry point: it exists for those callers only.
 *
 * B is row-major, so an unaligned A is always read in row classes and never
 * copied. A B whose base or row pitch is not a multiple of 16 bytes is
 * staged into one fixed, file-scope device array of
 * MPGEMM_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU which loads this
 * library holds until the process exits: K rows of round_up(N, 8) halves,
 * rounded up to 256 bytes, at most 16 MiB (e.g. K = 8192 with N up to 1024).
 * Beyond that the call returns MPGEMM_ERR_SCRATCH_LIMIT and enqueues
 * nothing; an aligned B needs no scratch and has no size limit beyond
 * mpgemm_run's.
 *
 * The first call on each device (with that device current) looks up the
 * array's device address and sets the kernels' shared-memory limits; make
 * that first call before any stream capture. If that set-up fails (for
 * example on a CUDA error left pending by other code), the call returns the
 * error and the next call tries the set-up again. All calls share the one array
 * and the work is stream-ordered only: calls whose work overlaps on the GPU
 * (different streams, or several host threads) race on the scratch and must
 * be serialised by the caller. A bounded device wait that gives up is
 * recorded only in the array's status words, not returned (use mpgemm_run
 * and mpgemm_sync_status where such reports are needed). Other arguments,
 * return codes and asynchrony are those of mpgemm_run. */
#define MPGEMM_NOALLOC_SCRATCH_BYTES (16ll * 1024 * 1024)
mpgemm_status_t mpgemm_run_noalloc(int64_t M, int64_t N, int64_t K,
                                   float alpha, const void* A, int64_t lda,
                                   const void* B, int64_t ldb,
                                   float beta, float* C, int64_t ldc, void* stream);

/* Measurement utility behind the theoretical tensor peak. The roofline of
 * "02_mixed_precision_gemm" README ("Experimental Setup") takes the dense
 * tensor peak as MACs per SM per clock x SMs x 2 x clock; this pins the per-SM
 * factor on the current device. `ctas` CTAs (use the SM count: each CTA
 * takes more than half an SM's shared memory, so one runs per SM) each issue
 * `mmas` back-to-back kind::f16 MMAs of M = 128, N = 256, K = 16 (FP16 x FP16
 * -> FP32, 1,048,576 FLOP each) from one thread, with no loads, and time them
 * with the SM cycle counter. `out` is a device array of 2 * ctas uint64_t:
 * out[2c] = cycles from the first issue to the last completion in CTA c,
 * out[2c + 1] = 1, or 0 if that CTA's bounded wait for the completion gave
 * up. FLOP per cycle per SM = 1048576 * mmas / out[2c]. Asynchronous on
 * `stream`; synchronise before reading `out`. Needs no handle and allocates
 * nothing. ctas in 1..65535, mmas in 4..4194304, `out` 8-byte aligned, else
 * MPGEMM_ERR_INVALID_VALUE; MPGEMM_ERR_UNSUPPORTED_DEVICE unless the
 * current device is compute capability 10.3. */
mpgemm_status_t mpgemm_probe_mma_rate(int32_t ctas, int32_t mmas, uint64_t* out, void* stream);

/* A static description of a status code. Never NULL. (No page defines this
 * call: it names the codes above.) */
const char* mpgemm_status_string(mpgemm_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* MPGEMM_H */
