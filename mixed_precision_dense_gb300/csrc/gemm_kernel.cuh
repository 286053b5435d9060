// The tensor-core pass of C = alpha*A*B + beta*C for sm_103a.
//
// Persistent CTAs walk the output in tiles. Each CTA has warps with fixed
// roles:
//   warp 0      load warp: one lane issues TMA loads of A (128 x 64, K-major)
//               and B (64 x 64 boxes: N-major when B is row-major, K-major
//               when B is column-major) into a ring of shared-memory stages;
//               rows, columns and K past the matrix edge arrive as zeros (TMA
//               out-of-bounds fill), which replaces the padding and guarded
//               tail loads of "Day 80, Capstone 4: a tensor-core GEMM"
//               ("Faded practice", practice 3; "Common failures").
//   warp 1      MMA warp: allocates tensor memory; one lane issues
//               tcgen05.mma (K = 16 per instruction, FP16 x FP16 -> FP32) and
//               frees each stage with tcgen05.commit.
//   warps 2-9   epilogue, two warps per 32 accumulator rows, each taking
//               half of the columns: each
//               warp reads its 32 accumulator rows with tcgen05.ld (32x32b:
//               TMEM lane = row) 32 columns at a time, applies alpha in FP32
//               and writes the 32 x 32 chunk into its own swizzled shared
//               buffer; from there either a tiled TMA store writes it to C
//               (beta == 0 and a TMA-addressable C), or each lane stores one
//               column (128 contiguous bytes per warp store instruction),
//               adding beta * C, or adding atomically for split-K; rows and
//               columns past M and N are masked, so any M, N and ldc work.
//               While it works on tile i, the MMAs of tile i+1 run into the
//               other accumulator buffer (or into the parts already drained).
//   warp 10     (CTA-pair tiles) a second MMA warp, the one after the
//               epilogue warps: for 256 x 512 tiles warp 1 issues the MMAs of
//               the first half of the accumulator's columns and this warp
//               those of the second; for 256 x 256 tiles the two take
//               alternate k-blocks, each at the full width, in a fixed order
//               (each thread issues its k-block only after the other thread
//               has issued the previous one; see TileConfig::KSPLIT). The
//               tensor pipe queues only about one MMA ahead of an issuing
//               thread, and each barrier wait stalls that thread; with two
//               issuers one keeps the pipe fed while the other waits
//               (measured: full MMA rate with two issuers, about 60 % with
//               one, for one barrier test per four MMAs).
//
// Two shapes of the same pipeline:
//   single  one CTA per tile of 128 x BN (BN = 128 or 256), tcgen05.mma with
//           cta_group::1, M = 128, N = 64 * ceil(valid columns / 64), two
//           accumulator buffers; or BN = 320 (N from 257 to 320 in one tile
//           column, so that every row block of A is read once), two
//           instructions per K step (N = 256 and N = 64) into one
//           accumulator buffer whose two parts are handed back one by one;
//   pair    a cluster of two CTAs per tile of 256 x BN (BN = 256, 320, 384
//           or 512): each CTA loads its own 128 rows of A and its own half of
//           the B columns of every accumulator part; the even CTA issues
//           tcgen05.mma with cta_group::2 (M = 256; N = 256, the full width
//           of a 256 x 256 tile, or per part of a wider tile: 256 + 64, 256
//           + 128, 256 + 256) over both CTAs' shared memory, and each CTA's
//           tensor memory receives its own 128 rows of the accumulator. Per
//           SM the 256 x 256 tile moves a third less operand data per FLOP
//           than the single 128 x 256 shape, the 256 x 512 tile half as
//           much. The 384- and 512-wide accumulators leave room for one
//           buffer, whose parts go back to their MMA threads one by one as
//           the epilogue drains them; the 320-wide one alternates two
//           staggered layouts (TileConfig::STAGGER).
//
// A stage holds one or two 64-wide k-blocks (TileConfig::KPS). The pairs of
// 256 to 384 columns can also walk the problem in stream-K ranges (one
// contiguous range of k-blocks per pair, GemmParams::sk_units) instead of
// whole tiles.

// The staged-tile reuse, asynchronous copies and block rasterisation that the
// pages build up with WMMA ("Day 80", "Worked path"; "02_mixed_precision_gemm"
// README, "Summary": cp.async double buffering and cross-block L2 reuse) map
// onto this design as: the tile held in shared memory and consumed by one
// MMA thread, the multistage TMA + mbarrier ring, and grouped rasterisation of
// the persistent tile walk.
//
// Every wait is bounded: if a barrier does not complete within the limit, the
// thread records the fact in the status words, raises a CTA-wide abort flag,
// lets its own in-flight copies and MMAs drain (again bounded), and the CTA
// releases its tensor memory and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace mpgemm {

// A is read through one tensor map per "row class". Usually there is one
// class holding every row. When A's rows do not start on 16-byte boundaries
// (an odd lda, say), the rows whose start addresses agree modulo U (U = 16,
// or U = 128: one L2 line) form a class: rows i = r (mod P), with P * lda * 2
// a multiple of U, so TMA can read them from the U-aligned address at or
// below row r, where they sit shifted right by a_shift(r) elements (up to 7,
// or up to 63). A tile then holds 128 rows of one class, and the matching B
// rows are fetched a_shift(r) rows earlier (rows before 0 arrive as zeros).
// With U = 128 every box row of A is one whole L2 line (measured on GB300,
// 65536 x 257 x 4093: rows starting mid-line cost 7 % at this size).
// P <= 8 for U = 16; U = 128 takes up to 64 classes, whose 8 KB of tensor
// maps only the tall-skinny kernels carry (TileConfig::A_CLASSES): larger
// kernel parameters cost the small calls about 0.2-0.5 us per launch.
constexpr int kMaxAClasses = 64;
// The kernels with room for 8 classes read each class's geometry from
// tables of 8 (the 64-class ones compute it: GemmParams; tables of 64, or
// the closed form in the 8-class kernels, cost the 256 x 384 pair 60 more
// bytes of spilled registers).
constexpr int kTableAClasses = 8;

// Most ranges of a stream-K walk (one per CTA pair).
constexpr int kMaxSkRanges = 128;

// Most CTAs (K slices) of a tile's cluster in the cluster split-K (the
// portable cluster size).
constexpr int kMaxClusterSlices = 8;

// The tensor maps of A (one per row class, room for NC classes), of C
// (FP32, 32 x 32 boxes, 128-byte swizzle; used only when GemmParams::c_tma
// is set) and of B in narrow boxes (used only by 256 x 288 and 256 x 320
// pair tiles).
template <int NC>
struct TensorMapsT {
    CUtensorMap a[NC];
    CUtensorMap c;
    CUtensorMap b_tail;   // B in 16- or 32-column boxes (32- or 64-byte swizzle): the narrow last part
};
using TensorMaps = TensorMapsT<kMaxAClasses>;

struct GemmParams {
    int32_t M, N, K;
    // Row classes of A (P of them; P = 1: every row, no shift). With M = P q
    // + m, classes r < m hold q + 1 rows (a_tiles_hi M-tiles), the others q
    // (a_tiles_lo); the M-tiles of class 0 come first, then those of class
    // 1, and so on. Class r's rows sit a_shift(r) = ((a_off0 + r a_step) mod
    // a_unit) / 2 elements right of the aligned address its tensor map
    // starts at (a_off0: A's address mod a_unit; a_step: 2 lda mod a_unit).
    int32_t a_classes;                  // P >= 1
    int32_t a_unit, a_off0, a_step;
    int32_t a_rem;                      // m
    int32_t a_rows_hi, a_rows_lo;       // q + 1, q
    int32_t a_tiles_hi, a_tiles_lo;
    // the same as tables, for P <= 8: shift, rows and first M-tile of class r
    int32_t a_shift[kTableAClasses];
    int32_t a_class_rows[kTableAClasses];
    int32_t a_class_first_tile[kTableAClasses + 1];
    int32_t m_tiles, n_tiles, k_blocks;   // tiles counted in units of the kernel's tile
    int32_t tiles;
    int32_t tail_start;     // tiles from here on (raster order) are done as two half-width items
    int32_t items;          // work items: tail_start + 2 * (tiles - tail_start), or tiles * k_splits
    int32_t k_splits;       // > 1: each tile's K range is cut into k_splits slices whose partial
    int32_t kb_per_split;   //      products are added into C (which already holds beta * C)
    int32_t raster_group;
    float alpha, beta;
    float* C;
    int64_t ldc;
    int32_t* status;        // {code, role, block, detail}
    uint64_t wait_limit_ns;
    int32_t test_stall;     // 1: the load warp issues nothing (timeout test)
    int32_t keep_a;         // L2 hints: 2 = keep both (evict-last), 1 = keep A (evict B first),
                            // 0 = keep B (evict A first)
    int32_t c_tma;          // 1: C is written through TensorMaps::c: TMA stores (beta == 0), or
                            //    TMA reduce-adds of split-K slices; one row class, C and ldc
                            //    16-byte aligned, N a multiple of 4
    int32_t acc16;          // 1: FP16 accumulators (the study variant; the product path is FP32)
    int32_t overlap_prepass;  // 1: launched right after this library's pass over C (C = beta * C
                              //    before split-K slices add into it): only the epilogue warps,
                              //    which write C, wait for it; the loads and MMAs start at once
    // Stream-K walk (sk_units > 0): the tiles' k-blocks, tile after tile in
    // raster order, are cut into sk_ranges contiguous ranges, range r being
    // [sk_start[r], sk_start[r + 1]) (at least one tile's k-blocks each), one
    // per persistent CTA (pair).
    // A tile cut between ranges r and r + 1 is written twice, in a fixed
    // order: range r + 1 does the tile's last k-blocks first and writes
    // C = alpha * (their sum) + beta * C, then publishes sk_epoch in its
    // flags; range r, whose last item holds the tile's first k-blocks, adds
    // alpha * (their sum) onto that C after it has seen the flag.
    int32_t sk_units;       // tiles * k_blocks (below 2^31), or 0
    int32_t sk_ranges;
    int32_t sk_epoch;       // this call's flag value (never 0)
    int32_t* sk_flags;      // [sk_ranges][CTAS][epilogue warps]: each epilogue warp publishes
                            // its own rows and columns of the tile
    int32_t sk_start[kMaxSkRanges + 1];
};

enum : int32_t { kRoleLoad = 1, kRoleMma = 2, kRoleEpilogue = 3 };
enum : int32_t { kStatusTimeout = 1 };

template <int BN_, int STAGES_, bool PAIR_, bool B_KMAJOR_ = false, int ISSUERS_ = (BN_ == 512 ? 2 : 1), int KPS_ = 1,
          bool CSPLIT_ = false>
struct TileConfig {
    static constexpr bool PAIR = PAIR_;
    // Split-K in clusters (one-CTA 128 x 128 tiles): the k_splits CTAs of a
    // cluster (GemmParams::k_splits of them, launched as one cluster per
    // tile) each sum one slice of K into their own accumulator, write it to
    // shared memory (over the idle ring) and, after a cluster barrier, each
    // sums its share of the tile's rows over every CTA's partial through
    // distributed shared memory, in CTA order, and writes C once: no pass
    // over C first, no atomics, the same bits on every call.
    static constexpr bool CSPLIT = CSPLIT_;
    // B column-major ([N, K] rows of K): a K-major operand like A. Its 64-row
    // boxes stack in shared memory exactly like the 64-column boxes of a
    // row-major B, so the ring layout is the same; only the box coordinates,
    // the shared-memory descriptor and the instruction's B-major bit differ.
    static constexpr bool B_KMAJOR = B_KMAJOR_;
    static constexpr int CTAS = PAIR ? 2 : 1;
    static constexpr int BM = 128;                     // accumulator rows per CTA
    static constexpr int TILE_M = BM * CTAS;           // rows per output tile
    static constexpr int BN = BN_;                     // columns per output tile
    static constexpr int B_COLS = BN / CTAS;           // columns of B each CTA loads
    static constexpr int BK = 64;                      // 64 halves = one 128-byte swizzle row
    // 64-wide k-blocks per pipeline stage: each stage holds KPS of them, A's
    // and B's boxes for each one after the other, and the kernel's k-block
    // unit (k_blocks, split-K slices, stream-K ranges) is a whole stage, SK
    // wide. Two per stage: one barrier round trip per 128 k, and each row of
    // A read 256 contiguous bytes at a time (a probe streaming the
    // tall-skinny pattern, no MMA: A from DRAM 4.2-4.6 TB/s with one per
    // stage, 5.3-5.5 TB/s with two)
    static constexpr int KPS = KPS_;
    static constexpr int SK = BK * KPS;
    static constexpr int STAGES = STAGES_;
    // threads issuing MMAs: one, or two. With two, a 512-wide tile gives
    // each issuer one part (a 256-column range) of the accumulator; a
    // 256-wide tile gives them alternate k-blocks instead (KSPLIT), each
    // issuing the full width (N = 256 instructions, twice as long as N = 128
    // ones, so the pipe holds twice the work ahead of each thread) into the
    // same accumulator. Their k-blocks are handed over in a strict order:
    // after issuing a k-block's MMAs (and committing its stage) a thread
    // executes tcgen05.fence::before_thread_sync and arrives on the stage's
    // hand-over barrier; the other thread waits on it, executes
    // tcgen05.fence::after_thread_sync and only then issues the next
    // k-block. The PTX ISA's memory consistency model for tcgen05 makes two
    // tcgen05.mma with the same accumulator, cta_group and shape a pipelined
    // pair, executed in the order they were issued, and the fence pair
    // around an arrive/wait carries that order from one thread to the other,
    // so the accumulator receives k-block 0, 1, 2, ... one after the other
    // without either thread waiting for MMAs to complete
    static constexpr int ISSUERS = ISSUERS_;
    static constexpr bool KSPLIT = ISSUERS == 2 && BN_ <= 256;
    // one MMA instruction covers SUB_N columns: BN, except that a tile wider
    // than 256 takes two instructions per K step, of 256 columns and of the
    // rest (256 for 512-wide pair tiles, 128 for 384-wide ones, 64 or 32 for
    // 320- or 288-wide ones)
    static constexpr int SUB_N = BN > 256 ? 256 : BN;
    static constexpr int SUBS = (BN + SUB_N - 1) / SUB_N;
    // columns of the last part; a pair CTA holds half of them. The last part
    // of a 320-wide pair is 64 columns, each CTA loading its 32 as one 4 KB
    // box in the 64-byte swizzle; that of a 288-wide pair 32 columns, 16 per
    // CTA in a 2 KB box in the 32-byte swizzle (row-major B only). For N =
    // 257 (one valid column there) the narrower part took 2 % off 65536 x 257
    // x 4093 and makes room for three stages of two k-blocks.
    static constexpr int TAIL_N = BN - (SUBS - 1) * SUB_N;
    static constexpr bool NARROW_TAIL = PAIR && (TAIL_N == 64 || TAIL_N == 32);
    // two accumulator buffers (the epilogue of tile i overlaps the MMAs of
    // tile i+1) when they fit in the 512 columns of tensor memory, else one,
    // whose SUBS parts are handed back one by one. A 320- or 288-wide pair
    // tile (STAGGER) alternates between two layouts of its 256-column part
    // and its last part (64 or 32 columns, in a 64-column slot) in the 512
    // columns, which overlap only by 64 columns each way:
    //   even items: 256-column part at column 0,   last part at 256
    //   odd items:  256-column part at column 256, last part at 0
    // Its epilogue hands back three parts in this order: the last part, the
    // first 64 columns of the 256-column part, and the other 192. The next
    // item's 256-column MMAs wait only for the first of them, its last-part
    // MMAs for the second; the 192 columns are drained while the next item's
    // MMAs run (one buffer of 320 columns made them wait for the whole
    // 256-column part).
    static constexpr bool STAGGER = NARROW_TAIL;
    static constexpr int ACC_BUFS = (STAGGER || 2 * BN <= 512) ? 2 : 1;
    static constexpr int RELEASE_PARTS = STAGGER ? 3 : (ACC_BUFS == 1 ? SUBS : 1);
    // B boxes (64 columns) per part held by one CTA: a pair CTA holds half
    // of every part's columns
    static constexpr int ATOMS_PER_PART = SUB_N / (PAIR ? 128 : 64);
    static constexpr int A_SUB_BYTES = BM * BK * 2;    // one 64-wide k-block of A: 16 KB
    static constexpr int A_BYTES = A_SUB_BYTES * KPS;
    static constexpr int B_ATOM_BYTES = BK * 64 * 2;   // one 64-column box of B: 8 KB
    static constexpr int B_SUB_BYTES = BK * B_COLS * 2;   // B of one 64-wide k-block
    static constexpr int B_BYTES = B_SUB_BYTES * KPS;
    static constexpr int B_TAIL_BYTES = BK * (TAIL_N / 2) * 2;   // one narrow box: a CTA's tail columns, 64 K-rows
    // epilogue warps: 8, two per 32 tensor-memory lanes, each taking half of
    // every part's columns. The 256 x 512 tile's single accumulator is
    // drained while the MMAs of the next tile wait, and the last tile of
    // every CTA is drained after its MMAs end; two warps per lane quarter
    // halve both (measured against four warps: 9-12 % less time per call
    // for GEMMs of one or two tiles per CTA)
    static constexpr int EPI_WARPS = 8;
    // the stream-K walk (GemmParams::sk_units) is built into the CTA-pair
    // shapes of at most 384 columns, those that run tall-skinny problems of
    // a few waves of tiles
    static constexpr bool STREAM_K = PAIR && BN <= 384;
    // the beta * C epilogue reads a chunk's 32 rows from shared memory
    // before storing any (not in 256 x 384 pairs, whose registers it spills:
    // 100 bytes, 65536 x 384 x 4096 200.0 -> 203.9 us)
    static constexpr bool EPI_BATCH_LOADS = BN != 384;
    // chunks of 32 accumulator columns, or (EPI_COLS 16: the 288-wide pair
    // with three stages of two k-blocks, which leave 22 KB for the buffers) of
    // 16, each through its warp's buffer of 32 rows (4 or 2 KB, 128- or
    // 64-byte swizzle, which TMA stores of 32 x 32 or 32 x 16 boxes read)
    static constexpr int EPI_COLS = (PAIR && BN == 288 && KPS == 2) ? 16 : 32;
    static constexpr int EPI_CHUNK_BYTES = 32 * EPI_COLS * 4;  // one warp's chunk buffer
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_CHUNK_BYTES;
    // row classes of A the kernel's parameters hold room for (see
    // kMaxAClasses): 64 for the row-major pairs of 288 and 320 columns of
    // one k-block per stage, which run the tall-skinny, memory-bound
    // problems with A in row classes, 8 for the rest
    static constexpr int A_CLASSES = (PAIR && !B_KMAJOR && (BN == 288 || BN == 320) && KPS == 1) ? kMaxAClasses : 8;
    // (allocations are powers of two: a 320-column accumulator takes 512)
    static constexpr int TMEM_COLS = (STAGGER || ACC_BUFS * BN > 256) ? 512 : 256;
    // full and empty per stage; accumulator full per buffer; accumulator
    // empty per buffer and part; k-block handed over per stage (KSPLIT)
    static constexpr int NUM_BARRIERS = 3 * STAGES + ACC_BUFS + ACC_BUFS * RELEASE_PARTS;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARRIERS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
    static constexpr int THREADS = 32 * (2 + EPI_WARPS + ISSUERS - 1);
    static_assert(BN == 128 || BN == 256 || BN == 320 || (PAIR && (BN == 288 || BN == 384 || BN == 512)), "tile width");
    static_assert(!NARROW_TAIL || (!B_KMAJOR && ISSUERS == 2), "narrow last part: row-major B, one issuer per part");
    static_assert(STAGGER ? ((BN == 320 || BN == 288) && SUB_N == 256) : ACC_BUFS * BN <= TMEM_COLS,
                  "accumulators fit the tensor memory allocated");
    static_assert(!PAIR || BN >= 256, "pair tiles are 256 x 256, 256 x 288, 256 x 320, 256 x 384 or 256 x 512");
    static_assert(ISSUERS == 1 || ISSUERS == SUBS || (KSPLIT && SUBS == 1), "one issuer, one per part, or two by k-block");
    static_assert(SUB_N >= (PAIR ? 128 : 64) && ATOMS_PER_PART >= 1, "parts hold whole B boxes");
    static_assert(A_SUB_BYTES % 1024 == 0 && B_SUB_BYTES % 1024 == 0, "stage alignment");
    static_assert(KPS == 1 || KPS == 2, "k-blocks per stage");
    static_assert(OFF_EPI % 1024 == 0, "chunk buffers are 1024-byte aligned (128-byte swizzle atoms)");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "tensor memory allocation");
    static_assert((BN % 64 == 0 || NARROW_TAIL) && (TAIL_N % (PAIR ? 128 : 64) == 0 || NARROW_TAIL),
                  "the last part holds whole B boxes");
    static_assert(A_CLASSES == 8 || A_CLASSES == kMaxAClasses, "row-class capacities");
    static_assert(!CSPLIT || (!PAIR && BN == 128 && STAGES * (A_BYTES + B_BYTES) >= 128 * 128 * 4),
                  "cluster split-K: one-CTA 128 x 128 tiles, the partial accumulator fits the ring");
};

// M-tile mb -> (row class r, first class row j0 of the tile), in a kernel
// with room for NC classes.
template <int TILE_M, int NC>
__device__ __forceinline__ void a_class_of(const GemmParams& p, int32_t mb, int32_t& r, int32_t& j0) {
    if constexpr (NC <= kTableAClasses) {
        r = 0;
        while (r + 1 < p.a_classes && mb >= p.a_class_first_tile[r + 1]) ++r;
        j0 = (mb - p.a_class_first_tile[r]) * TILE_M;
        return;
    }
    const int32_t hi_tiles = p.a_rem * p.a_tiles_hi;
    int32_t t;
    if (mb < hi_tiles) {
        r = mb / p.a_tiles_hi;
        t = mb - r * p.a_tiles_hi;
    } else {
        const int32_t q = (mb - hi_tiles) / p.a_tiles_lo;
        r = p.a_rem + q;
        t = mb - hi_tiles - q * p.a_tiles_lo;
    }
    j0 = t * TILE_M;
}
// elements before the rows of class r, and the rows it holds
template <int NC>
__device__ __forceinline__ int32_t a_shift_of(const GemmParams& p, int32_t r) {
    if constexpr (NC <= kTableAClasses) return p.a_shift[r];
    return ((p.a_off0 + r * p.a_step) & (p.a_unit - 1)) >> 1;   // a_unit: 16 or 128
}
template <int NC>
__device__ __forceinline__ int32_t a_rows_of(const GemmParams& p, int32_t r) {
    if constexpr (NC <= kTableAClasses) return p.a_class_rows[r];
    return r < p.a_rem ? p.a_rows_hi : p.a_rows_lo;
}

// Zero elements [16 j, 16 j + d) (d = 1..15) of the first `rows` rows of a
// 128-row A tile in the 128-byte-swizzled layout (16-byte chunk c of row t
// sits at chunk c ^ (t & 7)). These are the last of the a_shift = 16 j + d
// columns that lie before the rows' first element; the MMAs skip the
// 16-wide K slices below 16 j altogether. The matching B rows are zero, but
// the bytes there are arbitrary and could hold NaN or Inf. Rows past the
// matrix arrived as zeros already. At most four plain stores (16, 8, 4 and
// 2 bytes) per row, none of which waits for a load: this runs on the MMA
// thread before the tile's first instructions (a read-modify-write of every
// row there took about 8 K cycles on GB300).
struct LeadStores {
    int32_t c16, c;          // chunk of the 16-byte store (if s16), chunk of the partial stores
    bool s16, s8, s4, s2;
    int32_t o4, o2;          // offsets of the 4- and 2-byte stores within chunk c
};
__device__ __forceinline__ LeadStores lead_stores(int32_t j, int32_t d) {
    LeadStores z;
    z.s16 = d >= 8;
    z.c16 = 2 * j;
    z.c = 2 * j + (z.s16 ? 1 : 0);
    const int32_t part = d & 7;
    z.s8 = part >= 4;
    z.s4 = (part & 2) != 0;
    z.s2 = (part & 1) != 0;
    z.o4 = z.s8 ? 8 : 0;
    z.o2 = z.o4 + (z.s4 ? 4 : 0);
    return z;
}

__device__ __forceinline__ void zero_leading_columns(uint8_t* tile, int32_t j, int32_t d, int32_t rows) {
    const LeadStores z = lead_stores(j, d);
    rows = min(rows, 128);
#pragma unroll 8
    for (int32_t t = 0; t < rows; ++t) {
        uint8_t* row = tile + t * 128;
        if (z.s16) *reinterpret_cast<uint4*>(row + ((z.c16 ^ (t & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        uint8_t* q = row + ((z.c ^ (t & 7)) << 4);
        if (z.s8) *reinterpret_cast<uint64_t*>(q) = 0ull;
        if (z.s4) *reinterpret_cast<uint32_t*>(q + z.o4) = 0u;
        if (z.s2) *reinterpret_cast<uint16_t*>(q + z.o2) = static_cast<uint16_t>(0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The same for the A tile of the other CTA of a pair, written through
// distributed shared memory (tile_c: the tile's cluster address), then
// ordered before this thread's later tensor-core reads of it.
__device__ __forceinline__ void zero_leading_columns_peer(uint32_t tile_c, int32_t j, int32_t d, int32_t rows) {
    const LeadStores z = lead_stores(j, d);
    rows = min(rows, 128);
#pragma unroll 8
    for (int32_t t = 0; t < rows; ++t) {
        const uint32_t row = tile_c + static_cast<uint32_t>(t * 128);
        if (z.s16) {
            const uint32_t q16 = row + static_cast<uint32_t>((z.c16 ^ (t & 7)) << 4);
            ptx::st_cluster_u64(q16, 0ull);
            ptx::st_cluster_u64(q16 + 8, 0ull);
        }
        const uint32_t q = row + static_cast<uint32_t>((z.c ^ (t & 7)) << 4);
        if (z.s8) ptx::st_cluster_u64(q, 0ull);
        if (z.s4) ptx::st_cluster_u32(q + static_cast<uint32_t>(z.o4), 0u);
        if (z.s2) ptx::st_cluster_u16(q + static_cast<uint32_t>(z.o2), static_cast<uint16_t>(0));
    }
    ptx::fence_proxy_async_cluster();
}

// Tile t of the persistent walk -> (m block, n block). Tiles are visited in
// bands of `raster_group` M-blocks: down the band for one N-block, then the
// next N-block, so CTAs running at the same time share A and B panels in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int32_t t, int32_t& mb,
                                            int32_t& nb) {
    const int32_t per_band = p.raster_group * p.n_tiles;
    const int32_t band = t / per_band;
    const int32_t first_m = band * p.raster_group;
    const int32_t rows = min(p.m_tiles - first_m, p.raster_group);
    const int32_t r = t - band * per_band;
    mb = first_m + r % rows;
    nb = r / rows;
}

// Work item i of the persistent walk: a whole tile of width BN, or, past
// tail_start, one half (BN / 2 columns) of a tile (splitting the last partial
// wave of tiles in halves lets it finish in half the time), or, with
// k_splits > 1, one slice of a tile's K range (when there are too few tiles
// to occupy the GPU).
struct WorkItem {
    int32_t mb;      // tile row block
    int32_t n0;      // first column
    int32_t width;   // columns: BN or BN / 2
    int32_t kb0, kb1;  // k-blocks [kb0, kb1)
    int32_t sk;      // stream-K: kSkWhole, or kSkFirst (the tile's first k-blocks: added
                     // onto C after the next range has written it) or kSkRest (its
                     // other k-blocks, written first)
    int32_t range;   // stream-K: the range the item belongs to
};
enum : int32_t { kSkWhole = 0, kSkFirst = 1, kSkRest = 2 };

template <int BN, bool STREAM_K>
__device__ __forceinline__ WorkItem work_item(const GemmParams& p, int32_t i) {
    if (STREAM_K && p.sk_units > 0) {
        // item j of range r (i = r + j * sk_ranges, as the CTAs walk)
        const int32_t r = i % p.sk_ranges, j = i / p.sk_ranges;
        const int32_t u0 = p.sk_start[r], u1 = p.sk_start[r + 1];
        const int32_t t0 = u0 / p.k_blocks;
        const int32_t t_last = (u1 - 1) / p.k_blocks;
        // The range's tiles in order, except that a last piece holding a
        // tile's first k-blocks (kSkFirst) goes before the range's last
        // whole tile: its epilogue then runs while that tile's MMAs do, and
        // every range ends on a whole tile's epilogue.
        const int32_t n = t_last - t0 + 1;
        const bool first_last = u1 - t_last * p.k_blocks < p.k_blocks;
        const bool swap = first_last && (n >= 3 || (n == 2 && u0 == t0 * p.k_blocks));
        const int32_t jn = (swap && j >= n - 2 && j < n) ? (2 * n - 3 - j) : j;
        const int32_t t = t0 + jn;
        WorkItem w;
        w.range = r;
        w.width = BN;
        w.sk = kSkWhole;
        if (t > t_last) {   // none: past the last column, skipped by every role
            w.mb = 0;
            w.n0 = p.N;
            w.kb0 = w.kb1 = 0;
            return w;
        }
        int32_t mb, nb;
        tile_coords(p, t, mb, nb);
        w.mb = mb;
        w.n0 = nb * BN;
        w.kb0 = t == t0 ? u0 - t0 * p.k_blocks : 0;
        w.kb1 = t == t_last ? u1 - t_last * p.k_blocks : p.k_blocks;
        w.sk = w.kb0 > 0 ? kSkRest : (w.kb1 < p.k_blocks ? kSkFirst : kSkWhole);
        return w;
    }
    if (p.k_splits > 1) {
        const int32_t t = i / p.k_splits;
        const int32_t slice = i - t * p.k_splits;
        int32_t mb, nb;
        tile_coords(p, t, mb, nb);
        WorkItem w;
        w.mb = mb;
        w.n0 = nb * BN;
        w.width = BN;
        w.kb0 = slice * p.kb_per_split;
        w.kb1 = min(w.kb0 + p.kb_per_split, p.k_blocks);
        w.sk = kSkWhole;
        w.range = 0;
        return w;
    }
    int32_t t = i, half = -1;
    if (i >= p.tail_start) {
        const int32_t h = i - p.tail_start;
        t = p.tail_start + h / 2;
        half = h % 2;
    }
    int32_t mb, nb;
    tile_coords(p, t, mb, nb);
    WorkItem w;
    w.mb = mb;
    w.n0 = nb * BN + (half > 0 ? BN / 2 : 0);
    w.width = half < 0 ? BN : BN / 2;
    w.kb0 = 0;
    w.kb1 = p.k_blocks;
    w.sk = kSkWhole;
    w.range = 0;
    return w;
}

// Columns of item w that the MMAs cover: the item's width cut down to the
// 64-column boxes (one CTA) or 128-column units (a pair: each CTA holds half
// of every part) that hold columns below N (a 320-wide pair's 64-column last
// part counts whole).
template <class Cfg>
__device__ __forceinline__ int32_t item_cols(const GemmParams& p, const WorkItem& w) {
    constexpr int32_t unit = 64 * Cfg::CTAS;
    return min(w.width, unit * ((p.N - w.n0 + unit - 1) / unit));
}

// Part h (in the order the epilogue hands parts back) of the accumulator of
// an item using buffer buf: its first tensor-memory column, its first column
// within the item, and its width (item_width when the whole accumulator is
// one part).
struct AccPart {
    int32_t tmem_col, out_col, width;
};

template <class Cfg>
__device__ __forceinline__ AccPart acc_part(int h, int buf, int32_t item_width) {
    if constexpr (Cfg::STAGGER) {
        const int32_t main = buf ? 256 : 0, narrow = buf ? 0 : 256;
        if (h == 0) return {narrow, 256, 64};
        if (h == 1) return {main, 0, 64};
        return {main + 64, 64, 192};
    } else {
        return {buf * Cfg::BN + h * Cfg::SUB_N, h * Cfg::SUB_N, Cfg::RELEASE_PARTS > 1 ? Cfg::SUB_N : item_width};
    }
}

struct Waiter {
    const GemmParams* p;
    volatile int32_t* abort_flag;

    // Spin until the phase of `bar` with parity `parity` completes. Returns
    // false if the limit passes or another thread of the CTA aborted.
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (true) {
            if (ptx::mbar_try_wait(bar, parity)) return true;
            if (*abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > p->wait_limit_ns) return false;
        }
    }

    // Bounded wait used while draining after an abort (ignores the flag).
    __device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t0 < p->wait_limit_ns) {
        }
    }

    __device__ __forceinline__ void fail(int32_t role, int32_t detail) const {
        *abort_flag = 1;
        volatile int32_t* s = p->status;
        if (s[0] == 0) {
            s[1] = role;
            s[2] = static_cast<int32_t>(blockIdx.x);
            s[3] = detail;
            __threadfence_system();
            s[0] = kStatusTimeout;
        }
        __threadfence_system();
    }
};

// One lane's column `col` of 32 consecutive rows of C (rows at or past `rows`
// and columns at or past N read as 0). The 32 loads are independent, so they
// are in flight together.
__device__ __forceinline__ void load_c_chunk(const float* c_rows, int64_t ldc, int32_t col, int32_t N,
                                             int32_t rows, float (&v)[32]) {
    const bool col_ok = col < N;
#pragma unroll
    for (int rr = 0; rr < 32; ++rr)
        v[rr] = (col_ok && rr < rows) ? __ldg(c_rows + static_cast<int64_t>(rr) * ldc + col) : 0.0f;
}

// An accumulator element as read from tensor memory: FP32, or (FP16
// accumulators) an FP16 value in the low 16 bits of the 32-bit column
// (measured layout for kind::f16 with an F16 D: one element per column).
__device__ __forceinline__ float acc_value(uint32_t word, int32_t acc16) {
    return acc16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(word & 0xFFFFu))) : __uint_as_float(word);
}

// Byte offset of element (row, col) in a warp's 32 x 32 FP32 chunk buffer:
// rows of 128 bytes whose 16-byte groups sit at position group ^ (row & 7),
// the layout of the tensor memory accelerator's 128-byte swizzle. A lane
// writing its row as eight 16-byte stores, and 32 lanes reading one element
// each of a row, both touch every bank once.
__device__ __forceinline__ uint32_t chunk_off(int row, int col) {
    return static_cast<uint32_t>(row * 128 + ((((col >> 2) ^ row) & 7) << 4) + (col & 3) * 4);
}

// The same for a 32 x 16 chunk (64-byte rows; 16-byte group g of row r at
// g ^ ((r >> 1) & 3)): a lane writing its row's 16 columns as four 16-byte
// stores, and 32 lanes reading 16 columns of two rows, touch every bank once.
__device__ __forceinline__ uint32_t narrow_off(int row, int col) {
    return static_cast<uint32_t>(row * 64 + ((((col >> 2) ^ (row >> 1)) & 3) << 4) + (col & 3) * 4);
}

// Byte offset of accumulator element (row, col) of a 128 x 128 FP32 partial
// (cluster split-K): 512-byte rows, each 128-byte segment swizzled like a
// chunk buffer, so that a lane writing 32 columns of its row as eight
// 16-byte stores, and 32 lanes reading 32 consecutive columns of a row, both
// touch every bank once.
__device__ __forceinline__ uint32_t partial_off(int row, int col) {
    return static_cast<uint32_t>(row * 512 + (col >> 5) * 128 + (((((col & 31) >> 2) ^ row) & 7) << 4) +
                                 (col & 3) * 4);
}

// One 32 x 32 chunk (accumulator words r, TMEM lane = row = lane) to C,
// without a beta * C term: alpha applied, into the warp's chunk buffer, then
// either a tiled TMA store (a TMA reduce-add for split-K) at C row row0,
// column col0 (p.c_tma; the tensor map clips rows and columns outside C) or
// one column per lane (128 contiguous bytes per warp store instruction;
// atomic adds for split-K).
// Stream-K (SK): items of a tile cut between two ranges are written
// through per-lane stores, and the tile's first k-blocks (sk == kSkFirst)
// add onto C.
template <bool SK>
__device__ __forceinline__ bool chunk_tma(const GemmParams& p, int32_t sk) {
    return p.c_tma && (!SK || sk == kSkWhole);
}
template <bool SK>
__device__ __forceinline__ bool chunk_accumulate(const GemmParams& p, int32_t sk) {
    return p.k_splits > 1 || (SK && sk == kSkFirst);
}

template <bool SK>
__device__ __forceinline__ void emit_chunk(const GemmParams& p, const CUtensorMap* tmap_c, const uint32_t (&r)[32],
                                           float* c_tile, int64_t row_stride, int32_t rows, int32_t row0,
                                           int32_t col0, uint32_t buf_s, int lane, int32_t sk) {
    const float alpha = p.alpha;
    if (chunk_tma<SK>(p, sk)) {
        // the previous chunk's TMA store must have read the buffer
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
        ptx::st_shared_v4(buf_s + chunk_off(lane, 4 * q), alpha * acc_value(r[4 * q], p.acc16),
                          alpha * acc_value(r[4 * q + 1], p.acc16), alpha * acc_value(r[4 * q + 2], p.acc16),
                          alpha * acc_value(r[4 * q + 3], p.acc16));
    if (chunk_tma<SK>(p, sk)) {
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            // split-K slices add into C (which already holds beta * C)
            if (chunk_accumulate<SK>(p, sk))
                ptx::tma_reduce_add_2d(tmap_c, buf_s, col0, row0);
            else
                ptx::tma_store_2d(tmap_c, buf_s, col0, row0);
            ptx::bulk_commit_group();
        }
        return;
    }
    __syncwarp();
    const int32_t col = col0 + lane;
    if (col < p.N) {
        float* cp = c_tile + col;
        if (chunk_accumulate<SK>(p, sk)) {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr)
                if (rr < rows)
                    atomicAdd(cp + static_cast<int64_t>(rr) * row_stride, ptx::ld_shared_f32(buf_s + chunk_off(rr, lane)));
        } else {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr)
                if (rr < rows) cp[static_cast<int64_t>(rr) * row_stride] = ptx::ld_shared_f32(buf_s + chunk_off(rr, lane));
        }
    }
    __syncwarp();
}

// The epilogue of one work item for one warp: 32 rows of C (the tensor
// memory lanes of this warp's quarter; t_row addresses them at the
// accumulator's first column), of which the first `rows` exist, and columns
// n0 .. n0+width-1; row0 is the C row of the first of them and c_tile +
// rr * row_stride addresses row rr. Without a beta * C term the chunks'
// tensor-memory loads go out two at a time, and release() (which hands this
// part of the accumulator back to the MMA warp) runs as soon as the last of
// them has completed, before the last chunks are written. With beta != 0,
// c_cur holds the first chunk's old C values (loaded while the MMAs still
// ran), each later chunk's C loads go out before the previous chunk is
// stored, and release() runs once the last chunk's tensor-memory load has
// completed, before that chunk is stored.
template <bool SK, bool BATCH, class Release>
__device__ __forceinline__ void store_tile(const GemmParams& p, const CUtensorMap* tmap_c, uint32_t t_row,
                                          float* c_tile, int64_t row_stride, int32_t rows, int32_t row0,
                                          int32_t n0, int32_t width, uint32_t buf_s, int lane,
                                          float (&c_cur)[32], int32_t sk, Release&& release) {
    const float alpha = p.alpha, beta = p.beta;
    // (stream-K: the tile's first k-blocks add onto C without reading it)
    const bool read_c = beta != 0.0f && p.k_splits <= 1 && (!SK || sk != kSkFirst);
    const int32_t chunks = (min(width, p.N - n0) + 31) / 32;
    if (!read_c) {
        for (int32_t c = 0; c < chunks; c += 2) {
            uint32_t r0[32], r1[32];
            const bool two = c + 1 < chunks;
            ptx::tmem_load_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r0);
            if (two) ptx::tmem_load_32x32b_x32(t_row + static_cast<uint32_t>((c + 1) * 32), r1);
            ptx::tmem_load_wait();
            ptx::tmem_regs_ready(r0);
            if (two) ptx::tmem_regs_ready(r1);
            if (c + 2 >= chunks) release();
            emit_chunk<SK>(p, tmap_c, r0, c_tile, row_stride, rows, row0, n0 + c * 32, buf_s, lane, sk);
            if (two) emit_chunk<SK>(p, tmap_c, r1, c_tile, row_stride, rows, row0, n0 + (c + 1) * 32, buf_s, lane, sk);
        }
        if (chunks <= 0) release();
        return;
    }
    const float* c_rows = c_tile;
    float c_next[32];
    for (int32_t c = 0; c < chunks; ++c) {
        uint32_t r[32];
        ptx::tmem_load_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
        if (c + 1 < chunks)
            load_c_chunk(c_rows, row_stride, n0 + (c + 1) * 32 + lane, p.N, rows, c_next);
        ptx::tmem_load_wait();
        ptx::tmem_regs_ready(r);
        if (c + 1 >= chunks) release();   // the part's last tensor-memory load has completed
#pragma unroll
        for (int q = 0; q < 8; ++q)
            ptx::st_shared_v4(buf_s + chunk_off(lane, 4 * q), alpha * acc_value(r[4 * q], p.acc16),
                              alpha * acc_value(r[4 * q + 1], p.acc16), alpha * acc_value(r[4 * q + 2], p.acc16),
                              alpha * acc_value(r[4 * q + 3], p.acc16));
        __syncwarp();
        const int32_t col = n0 + c * 32 + lane;
        if (col < p.N) {
            float* cp = c_tile + col;
            if constexpr (BATCH) {
                // the lane's 32 rows read from shared memory first, into the
                // registers that held the accumulator words: the loads issue
                // back to back instead of each waiting behind the previous
                // row's global store (65536 x 257 x 4093, beta 0.5: 171.7 ->
                // 169.3 us)
#pragma unroll
                for (int rr = 0; rr < 32; ++rr)
                    r[rr] = __float_as_uint(ptx::ld_shared_f32(buf_s + chunk_off(rr, lane)));
#pragma unroll
                for (int rr = 0; rr < 32; ++rr)
                    if (rr < rows)
                        cp[static_cast<int64_t>(rr) * row_stride] = fmaf(beta, c_cur[rr], __uint_as_float(r[rr]));
            } else {
#pragma unroll
                for (int rr = 0; rr < 32; ++rr)
                    if (rr < rows)
                        cp[static_cast<int64_t>(rr) * row_stride] =
                            fmaf(beta, c_cur[rr], ptx::ld_shared_f32(buf_s + chunk_off(rr, lane)));
            }
        }
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) c_cur[rr] = c_next[rr];
        __syncwarp();
    }
    if (chunks <= 0) release();
}

// 16-column chunks (TileConfig::EPI_COLS 16). A lane's part of a 32 x 16
// chunk whose first column is col0: column col0 + (lane & 15) of rows
// 2 i + (lane >> 4), i < 16 (two 64-byte row pieces per warp store
// instruction). load_c_chunk16 reads the old C values of those elements
// into v[0..15] (rows at or past `rows`, columns at or past N: 0).
__device__ __forceinline__ void load_c_chunk16(const float* c_rows, int64_t ldc, int32_t col0, int lane, int32_t N,
                                               int32_t rows, float (&v)[32]) {
    const int32_t rh = lane >> 4, col = col0 + (lane & 15);
    const bool col_ok = col < N;
    const float* q = c_rows + static_cast<int64_t>(rh) * ldc + col;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = (col_ok && 2 * i + rh < rows) ? __ldg(q + static_cast<int64_t>(2 * i) * ldc) : 0.0f;
}

// One 32 x 16 chunk (accumulator words r, TMEM lane = row = lane) to C
// without a beta * C term: alpha applied, through the warp's buffer (whose
// layout is the tensor memory accelerator's 64-byte swizzle), then either a
// tiled TMA store (reduce-add for split-K) of the 32 x 16 box at C row row0,
// column col0 (p.c_tma), or read back into r and stored (atomic adds for
// split-K or a stream-K first piece) lane by lane.
template <bool SK>
__device__ __forceinline__ void emit_chunk16(const GemmParams& p, const CUtensorMap* tmap_c, uint32_t (&r)[16],
                                             float* c_tile, int64_t row_stride, int32_t rows, int32_t row0,
                                             int32_t col0, uint32_t buf_s, int lane, int32_t sk) {
    const float alpha = p.alpha;
    if (chunk_tma<SK>(p, sk)) {
        // the previous chunk's TMA store must have read the buffer
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
        ptx::st_shared_v4(buf_s + narrow_off(lane, 4 * q), alpha * acc_value(r[4 * q], p.acc16),
                          alpha * acc_value(r[4 * q + 1], p.acc16), alpha * acc_value(r[4 * q + 2], p.acc16),
                          alpha * acc_value(r[4 * q + 3], p.acc16));
    if (chunk_tma<SK>(p, sk)) {
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (chunk_accumulate<SK>(p, sk))
                ptx::tma_reduce_add_2d(tmap_c, buf_s, col0, row0);
            else
                ptx::tma_store_2d(tmap_c, buf_s, col0, row0);
            ptx::bulk_commit_group();
        }
        return;
    }
    __syncwarp();
    const int32_t rh = lane >> 4, cl = lane & 15;
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(ptx::ld_shared_f32(buf_s + narrow_off(2 * i + rh, cl)));
    const int32_t col = col0 + cl;
    if (col < p.N) {
        float* cp = c_tile + col + static_cast<int64_t>(rh) * row_stride;
        const bool add = chunk_accumulate<SK>(p, sk);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (2 * i + rh < rows) {
                float* e = cp + static_cast<int64_t>(2 * i) * row_stride;
                if (add)
                    atomicAdd(e, __uint_as_float(r[i]));
                else
                    *e = __uint_as_float(r[i]);
            }
        }
    }
    __syncwarp();
}

// store_tile for 16-column chunks (the same contract): without beta * C the
// chunks' tensor-memory loads go out two at a time; with beta != 0, c_cur
// holds the first chunk's old C values (load_c_chunk16's order), and each
// later chunk's go out before the previous chunk is stored.
template <bool SK, class Release>
__device__ __forceinline__ void store_tile16(const GemmParams& p, const CUtensorMap* tmap_c, uint32_t t_row,
                                            float* c_tile, int64_t row_stride, int32_t rows, int32_t row0,
                                            int32_t n0, int32_t width, uint32_t buf_s, int lane,
                                            float (&c_cur)[32], int32_t sk, Release&& release) {
    const float alpha = p.alpha, beta = p.beta;
    const bool read_c = beta != 0.0f && p.k_splits <= 1 && (!SK || sk != kSkFirst);
    const int32_t chunks = (min(width, p.N - n0) + 15) / 16;
    if (!read_c) {
        for (int32_t c = 0; c < chunks; c += 2) {
            uint32_t r0[16], r1[16];
            const bool two = c + 1 < chunks;
            ptx::tmem_load_32x32b_x16(t_row + static_cast<uint32_t>(c * 16), r0);
            if (two) ptx::tmem_load_32x32b_x16(t_row + static_cast<uint32_t>((c + 1) * 16), r1);
            ptx::tmem_load_wait();
            ptx::tmem_regs_ready(r0);
            if (two) ptx::tmem_regs_ready(r1);
            if (c + 2 >= chunks) release();
            emit_chunk16<SK>(p, tmap_c, r0, c_tile, row_stride, rows, row0, n0 + c * 16, buf_s, lane, sk);
            if (two)
                emit_chunk16<SK>(p, tmap_c, r1, c_tile, row_stride, rows, row0, n0 + (c + 1) * 16, buf_s, lane, sk);
        }
        if (chunks <= 0) release();
        return;
    }
    const int32_t rh = lane >> 4, cl = lane & 15;
    float c_next[32];
    for (int32_t c = 0; c < chunks; ++c) {
        uint32_t r[16];
        ptx::tmem_load_32x32b_x16(t_row + static_cast<uint32_t>(c * 16), r);
        if (c + 1 < chunks) load_c_chunk16(c_tile, row_stride, n0 + (c + 1) * 16, lane, p.N, rows, c_next);
        ptx::tmem_load_wait();
        ptx::tmem_regs_ready(r);
        if (c + 1 >= chunks) release();   // the part's last tensor-memory load has completed
#pragma unroll
        for (int q = 0; q < 4; ++q)
            ptx::st_shared_v4(buf_s + narrow_off(lane, 4 * q), alpha * acc_value(r[4 * q], p.acc16),
                              alpha * acc_value(r[4 * q + 1], p.acc16), alpha * acc_value(r[4 * q + 2], p.acc16),
                              alpha * acc_value(r[4 * q + 3], p.acc16));
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(ptx::ld_shared_f32(buf_s + narrow_off(2 * i + rh, cl)));
        const int32_t col = n0 + c * 16 + cl;
        if (col < p.N) {
            float* cp = c_tile + col + static_cast<int64_t>(rh) * row_stride;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (2 * i + rh < rows)
                    cp[static_cast<int64_t>(2 * i) * row_stride] = fmaf(beta, c_cur[i], __uint_as_float(r[i]));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) c_cur[i] = c_next[i];
        __syncwarp();
    }
    if (chunks <= 0) release();
}

// Cluster split-K: CTA `rank` of the tile's cluster owns rows [r0, r1) of
// the 128-row tile (shares of R = ceil(128 / k_splits) rows, cut at the
// tile's last row); c_tile + row * row_stride addresses the tile's C row.
struct CsplitShare {
    int32_t n0, r0, r1;
    int64_t row_stride;
    float* c_tile;
};
template <class Cfg>
__device__ __forceinline__ CsplitShare csplit_share(const GemmParams& p) {
    const int32_t S = p.k_splits;
    const int32_t rank = static_cast<int32_t>(ptx::cluster_ctarank());
    int32_t mb, nb, cls, j0;
    tile_coords(p, static_cast<int32_t>(blockIdx.x) / S, mb, nb);
    a_class_of<Cfg::TILE_M, Cfg::A_CLASSES>(p, mb, cls, j0);
    const int32_t rows = min(Cfg::BM, a_rows_of<Cfg::A_CLASSES>(p, cls) - j0);
    const int32_t share = (Cfg::BM + S - 1) / S;
    CsplitShare c;
    c.n0 = nb * Cfg::BN;
    c.r0 = rank * share;
    c.r1 = min(rows, c.r0 + share);
    c.row_stride = static_cast<int64_t>(p.a_classes) * p.ldc;
    c.c_tile = p.C + (cls + static_cast<int64_t>(p.a_classes) * j0) * p.ldc;
    return c;
}

// Every warp of the CTA takes two rows of its share at a time, each lane
// columns lane, lane + 32, lane + 64 and lane + 96 of them; all the loads of
// the two rows (the k_splits partials through distributed shared memory, and
// the old C) go out before any is used. An element is the sum of the
// partials in CTA order, then alpha times it plus beta times the old C (beta
// == 0: C is not read).
template <class Cfg>
__device__ __forceinline__ void csplit_reduce(const GemmParams& p, uint32_t partial) {
    static_assert(Cfg::BN == 128, "four columns per lane");
    constexpr int NW = Cfg::THREADS / 32;
    const int32_t S = p.k_splits;
    const CsplitShare sh = csplit_share<Cfg>(p);
    const bool read_c = p.beta != 0.0f;
    uint32_t src[kMaxClusterSlices];
#pragma unroll
    for (int s = 0; s < kMaxClusterSlices; ++s)
        src[s] = ptx::mapa_shared(partial, static_cast<uint32_t>(s < S ? s : 0));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int32_t row = sh.r0 + warp; row < sh.r1; row += 2 * NW) {
        float v[kMaxClusterSlices][2][4], c_old[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int32_t r = row + rr * NW;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int32_t col = sh.n0 + q * 32 + lane;
                c_old[rr][q] = (read_c && r < sh.r1 && col < p.N)
                                   ? __ldg(sh.c_tile + static_cast<int64_t>(r) * sh.row_stride + col)
                                   : 0.0f;
            }
        }
#pragma unroll
        for (int s = 0; s < kMaxClusterSlices; ++s)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    v[s][rr][q] = (s < S && row + rr * NW < sh.r1)
                                      ? ptx::ld_cluster_f32(src[s] + partial_off(row + rr * NW, q * 32 + lane))
                                      : 0.0f;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int32_t r = row + rr * NW;
            if (r >= sh.r1) continue;
            float* c_row = sh.c_tile + static_cast<int64_t>(r) * sh.row_stride;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int32_t col = sh.n0 + q * 32 + lane;
                if (col >= p.N) continue;
                float sum = v[0][rr][q];
#pragma unroll
                for (int s = 1; s < kMaxClusterSlices; ++s)
                    if (s < S) sum += v[s][rr][q];
                const float out = p.alpha * sum;
                c_row[col] = read_c ? fmaf(p.beta, c_old[rr][q], out) : out;
            }
        }
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ TensorMapsT<Cfg::A_CLASSES> maps,
                   const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr bool PAIR = Cfg::PAIR;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw_addr);

    const uint32_t sA = base + Cfg::OFF_A;
    const uint32_t sB = base + Cfg::OFF_B;
    const uint32_t bar0 = base + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    constexpr int ACC_BUFS = Cfg::ACC_BUFS, RELEASE_PARTS = Cfg::RELEASE_PARTS;
    auto acc_full_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acc_empty_bar = [&](int b, int h) { return bar0 + 8u * (2 * STAGES + ACC_BUFS + b * RELEASE_PARTS + h); };
    // (KSPLIT) arrived on once the k-block held in stage s has been issued
    auto handed_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + ACC_BUFS + ACC_BUFS * RELEASE_PARTS + s); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Cfg::OFF_MISC);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + Cfg::OFF_MISC + 4);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const Waiter waiter{&p, abort_flag};
    // Pair: the even CTA of the cluster issues the MMAs and owns the barriers
    // both CTAs' loads and epilogues report to.
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    const int32_t first_item = PAIR ? static_cast<int32_t>(blockIdx.x / 2) : static_cast<int32_t>(blockIdx.x);
    const int32_t item_step = PAIR ? static_cast<int32_t>(gridDim.x / 2) : static_cast<int32_t>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), Cfg::KSPLIT ? 1 : Cfg::ISSUERS);   // one commit per issuer using it
            ptx::mbar_init(handed_bar(s), 1);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            ptx::mbar_init(acc_full_bar(b), Cfg::ISSUERS);
            for (int h = 0; h < RELEASE_PARTS; ++h) ptx::mbar_init(acc_empty_bar(b, h), Cfg::EPI_WARPS * Cfg::CTAS);
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int r = 0; r < min(p.a_classes, Cfg::A_CLASSES); ++r) ptx::prefetch_tensormap(&maps.a[r]);
        if (p.c_tma) ptx::prefetch_tensormap(&maps.c);
        if constexpr (Cfg::NARROW_TAIL) ptx::prefetch_tensormap(&maps.b_tail);
        ptx::prefetch_tensormap(&tmap_b);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), Cfg::TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(tmem_slot), Cfg::TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();   // peer barriers initialised before any remote use
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // The GEMM is launched with programmatic stream serialization: it may
    // start while the previous kernel of the stream (a staging or C-scaling
    // pass, or the previous GEMM) is still finishing, and everything above
    // (barriers, tensor memory, tensor-map prefetch) touches no global
    // memory. Every thread waits here until that kernel has completed and
    // its writes are visible; the next kernel may begin its own setup now.
    ptx::griddep_launch_dependents();
    // (after the library's own pass over C, which itself started only once
    // everything before it in the stream had completed, A and B are ready:
    // only C has to wait for that pass)
    if (!p.overlap_prepass || (warp >= 2 && warp < 2 + Cfg::EPI_WARPS)) ptx::griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ loads
        if (lane == 0) {
            // Both operands are loaded evict-last unless only one tile reads
            // them (keep_a, chosen by the host; C's stores are evict-first):
            // every panel is re-read by the other tiles of its wave, and
            // marking either operand evict-first cost L2 reuse (DRAM reads at
            // 8192^3: 845 MB per launch, against 1224 MB with B evict-first).
            const uint64_t pol_a = p.keep_a == 0 ? ptx::policy_evict_first() : ptx::policy_evict_last();
            const uint64_t pol_b = p.keep_a == 1 ? ptx::policy_evict_first() : ptx::policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0;               // stages this CTA armed with expect_tx
            uint32_t armed_parity = 0;        // parity of the last armed phase per stage
            bool ok = true;
            if (!p.test_stall) {
                for (int32_t i = first_item; ok && i < p.items; i += item_step) {
                    const WorkItem w = work_item<BN, Cfg::STREAM_K>(p, i);
                    if (w.n0 >= p.N) continue;   // a half tile wholly past the last column
                    // Pair: each MMA instruction covers sub_n columns of the
                    // item, and this CTA loads sub_n / 2 of them (its half) for
                    // each instruction, in 64-column boxes ("atoms"); atom a
                    // belongs to instruction a / per_sub.
                    const int32_t n_valid = item_cols<Cfg>(p, w);
                    int32_t cls, j0;
                    a_class_of<Cfg::TILE_M, Cfg::A_CLASSES>(p, w.mb, cls, j0);
                    const CUtensorMap* map_a = &maps.a[cls];
                    const int32_t a_row = j0 + static_cast<int32_t>(rank) * BM;   // class row
                    const int32_t b_shift = a_shift_of<Cfg::A_CLASSES>(p, cls);
                    // only the boxes that hold valid columns (a pair CTA holds
                    // half of every part's columns)
                    const int32_t n_atoms = n_valid / (64 * Cfg::CTAS);
                    const uint32_t bytes = (Cfg::A_BYTES + (n_valid / Cfg::CTAS) * Cfg::SK * 2) * Cfg::CTAS;
                    for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                        if (!waiter.wait(empty_bar(stage), phase ^ 1u)) {
                            waiter.fail(kRoleLoad, kb);
                            ok = false;
                            break;
                        }
                        if constexpr (PAIR) {
                            const uint32_t lead_full = ptx::mapa_shared(full_bar(stage), 0);
                            if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
                            // the stage's KPS k-blocks of A first (back to back: 64 * KPS
                            // contiguous halves of every row), then their B
#pragma unroll
                            for (int q = 0; q < Cfg::KPS; ++q)
                                ptx::tma_load_2d_pair(sA + stage * Cfg::A_BYTES + q * Cfg::A_SUB_BYTES, map_a, lead_full,
                                                      kb * Cfg::SK + q * BK, a_row, pol_a);
#pragma unroll
                            for (int q = 0; q < Cfg::KPS; ++q) {
                                const int32_t k0 = kb * Cfg::SK + q * BK;
                                // part h (an MMA instruction's columns): this CTA loads
                                // its half of them, in 64-column boxes from box h *
                                // ATOMS_PER_PART on
                                for (int32_t h = 0; h * Cfg::SUB_N < n_valid; ++h) {
                                    const int32_t half = min(Cfg::SUB_N, n_valid - h * Cfg::SUB_N) / 2;
                                    const int32_t c0 = w.n0 + h * Cfg::SUB_N + static_cast<int32_t>(rank) * half;
                                    const uint32_t dst = sB + stage * Cfg::B_BYTES + q * Cfg::B_SUB_BYTES +
                                                         h * Cfg::ATOMS_PER_PART * Cfg::B_ATOM_BYTES;
                                    if (Cfg::NARROW_TAIL && half == Cfg::TAIL_N / 2) {
                                        ptx::tma_load_2d_pair(dst, &maps.b_tail, lead_full, c0, k0 - b_shift, pol_b);
                                        continue;
                                    }
                                    for (int32_t a = 0; a * 64 < half; ++a) {
                                        const int32_t col = c0 + a * 64;
                                        ptx::tma_load_2d_pair(dst + a * Cfg::B_ATOM_BYTES, &tmap_b, lead_full,
                                                              Cfg::B_KMAJOR ? k0 : col, Cfg::B_KMAJOR ? col : k0 - b_shift,
                                                              pol_b);
                                    }
                                }
                            }
                        } else {
                            ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
#pragma unroll
                            for (int q = 0; q < Cfg::KPS; ++q)
                                ptx::tma_load_2d(sA + stage * Cfg::A_BYTES + q * Cfg::A_SUB_BYTES, map_a, full_bar(stage),
                                                 kb * Cfg::SK + q * BK, a_row, pol_a);
#pragma unroll
                            for (int q = 0; q < Cfg::KPS; ++q) {
                                const int32_t k0 = kb * Cfg::SK + q * BK;
                                for (int j = 0; j < n_atoms; ++j)
                                    ptx::tma_load_2d(sB + stage * Cfg::B_BYTES + q * Cfg::B_SUB_BYTES + j * Cfg::B_ATOM_BYTES,
                                                     &tmap_b, full_bar(stage), Cfg::B_KMAJOR ? k0 : w.n0 + j * 64,
                                                     Cfg::B_KMAJOR ? w.n0 + j * 64 : k0 - b_shift, pol_b);
                            }
                        }
                        if (rank == 0) {
                            armed |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        }
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                // Let the loads of every armed stage land before the CTA exits.
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s)) waiter.drain(full_bar(s), (armed_parity >> s) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1 || (Cfg::ISSUERS > 1 && warp == 2 + Cfg::EPI_WARPS)) {
        // ------------------------------------------------------------ MMA
        // Issuer `me` handles accumulator part `me` (all parts when there is
        // one issuer). Every issuer waits for every stage and commits it, so
        // a stage is freed only when all issuers' MMAs on it have completed;
        // an issuer with no part in an item (a half-width item) still does.
        // KSPLIT: issuer `me` takes the k-blocks whose running count g (over
        // all items of this CTA) has parity `me`, and commits only those;
        // k-block g is issued only after k-block g - 1 (the other thread's,
        // held in the previous stage) has been issued and handed over.
        const int me = warp == 1 ? 0 : 1;
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            auto next_stage = [&]() {
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            int32_t local = 0;
            bool ok = true;
            bool issued = false;
            int64_t walked = 0;   // k-blocks of the items before this one (KSPLIT)
            for (int32_t i = first_item; ok && i < p.items; i += item_step) {
                const WorkItem w = work_item<BN, Cfg::STREAM_K>(p, i);
                if (w.n0 >= p.N) continue;
                // columns the MMAs cover (the boxes wholly past N are skipped)
                // and the parts (instructions per K step) they fall into: part
                // h is columns [h SUB_N, h SUB_N + cols)
                const int32_t n_valid = item_cols<Cfg>(p, w);
                const int32_t n_parts = (n_valid + Cfg::SUB_N - 1) / Cfg::SUB_N;
                int32_t cls, j0;
                a_class_of<Cfg::TILE_M, Cfg::A_CLASSES>(p, w.mb, cls, j0);
                const int32_t lead_cols = a_shift_of<Cfg::A_CLASSES>(p, cls);   // columns before the rows' start
                const int32_t lead_rows = a_rows_of<Cfg::A_CLASSES>(p, cls) - j0;   // rows of the tile that exist
                // k-block 0 of the tile: its first lead_cols / 16 slices of 16
                // lie wholly before the rows' start and are not issued; the
                // rest of those columns are zeroed in shared memory
                const int32_t lead_k16 = lead_cols >> 4, lead_part = lead_cols & 15;
                const int buf = local % ACC_BUFS;
                const uint32_t acc_phase = (local / ACC_BUFS) & 1;
                if constexpr (RELEASE_PARTS == 1) {
                    if (!waiter.wait(acc_empty_bar(buf, 0), acc_phase ^ 1u)) {
                        waiter.fail(kRoleMma, -1);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                }
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(Cfg::STAGGER ? 0 : buf * BN);
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if constexpr (Cfg::KSPLIT) {
                        if (((walked + (kb - w.kb0)) & 1) != me) {   // the other issuer's k-block
                            next_stage();
                            continue;
                        }
                    }
                    if (!waiter.wait(full_bar(stage), phase)) {
                        waiter.fail(kRoleMma, kb);
                        ok = false;
                        break;
                    }
                    if constexpr (Cfg::KSPLIT) {
                        // wait until the other thread has issued k-block g - 1
                        // (stage g - 1 of the ring, the phase it had then). The
                        // barrier cannot move on by a second phase meanwhile:
                        // that thread issues k-block g - 1 + STAGES only after
                        // this one has issued g, ..., g - 2 + STAGES.
                        const int64_t g = walked + (kb - w.kb0);
                        if (g > 0) {
                            const int ps = stage == 0 ? STAGES - 1 : stage - 1;
                            const uint32_t pph = stage == 0 ? (phase ^ 1u) : phase;
                            if (!waiter.wait(handed_bar(ps), pph)) {
                                waiter.fail(kRoleMma, kb);
                                ok = false;
                                break;
                            }
                        }
                    }
                    ptx::tc_fence_after_sync();
                    if (kb == 0 && lead_part > 0) {
                        zero_leading_columns(gbase + Cfg::OFF_A + stage * Cfg::A_BYTES, lead_k16, lead_part, lead_rows);
                        // the other CTA of a pair holds the tile's next 128 rows
                        if constexpr (PAIR)
                            zero_leading_columns_peer(ptx::mapa_shared(sA + stage * Cfg::A_BYTES, 1), lead_k16,
                                                      lead_part, lead_rows - BM);
                    }
                    const int32_t skip16 = kb == 0 ? lead_k16 : 0;   // slices not issued
                    const uint32_t a_base = sA + stage * Cfg::A_BYTES;
                    const uint32_t b_base = sB + stage * Cfg::B_BYTES;
                    bool pending = false;   // MMAs issued from this stage
                    const int32_t h_begin = (Cfg::ISSUERS > 1 && !Cfg::KSPLIT) ? me : 0;
                    const int32_t h_end = (Cfg::ISSUERS > 1 && !Cfg::KSPLIT) ? min(me + 1, n_parts) : n_parts;
                    for (int32_t h = h_begin; ok && h < h_end; ++h) {
                        if constexpr (Cfg::STAGGER) {
                            // the first use of part h in this item: wait until the
                            // epilogue has read what overlaps it: the same part of
                            // the item before last (same layout; for the 256-column
                            // part its last-released third implies the others), and
                            // of the previous item (other layout) the 64 columns
                            // handed back first (256-column part) or second
                            // (64-column part)
                            if (kb == w.kb0) {
                                bool fine = true;
#pragma unroll 1
                                for (int q = 0; fine && q < (local > 0 ? 2 : 1); ++q)
                                    fine = q == 0 ? waiter.wait(acc_empty_bar(buf, h == 0 ? 2 : 0), acc_phase ^ 1u)
                                                  : waiter.wait(acc_empty_bar(buf ^ 1, h == 0 ? 0 : 1),
                                                                static_cast<uint32_t>((local - 1) / 2) & 1u);
                                if (!fine) {
                                    waiter.fail(kRoleMma, -1);
                                    ok = false;
                                    break;
                                }
                                ptx::tc_fence_after_sync();
                            }
                        } else if constexpr (RELEASE_PARTS > 1) {
                            // the first use of part h in this item: wait until the
                            // epilogue has read the previous item's part h
                            if (kb == w.kb0) {
                                if (!waiter.wait(acc_empty_bar(0, h), acc_phase ^ 1u)) {
                                    waiter.fail(kRoleMma, -1);
                                    ok = false;
                                    break;
                                }
                                ptx::tc_fence_after_sync();
                            }
                        }
                        // part h: SUB_N accumulator columns further, ATOMS_PER_PART
                        // B boxes further (a pair CTA holds half of each part's
                        // columns); D format bits 4-5: 1 = F32 accumulators,
                        // 0 = F16 (the study variant)
                        const int32_t part_cols = min(Cfg::SUB_N, n_valid - h * Cfg::SUB_N);
                        const uint32_t idesc = ptx::idesc_f16_f32(Cfg::TILE_M, part_cols, false, !Cfg::B_KMAJOR) &
                                               ~(p.acc16 ? (3u << 4) : 0u);
                        const uint32_t d_part =
                            d_tmem + static_cast<uint32_t>(Cfg::STAGGER ? ((h == 0) == (buf == 0) ? 0 : 256) : h * Cfg::SUB_N);
                        const uint32_t b_part =
                            b_base + static_cast<uint32_t>(h * Cfg::ATOMS_PER_PART * Cfg::B_ATOM_BYTES);
#pragma unroll
                        for (int k16 = 0; k16 < Cfg::SK / 16; ++k16) {
                            if (k16 < skip16) continue;
                            // (64-wide k-block q of the stage, its 16-wide slice kk)
                            const int q = k16 / (BK / 16), kk = k16 % (BK / 16);
                            const uint32_t b_q = b_part + static_cast<uint32_t>(q * Cfg::B_SUB_BYTES);
                            // A: K-major, 128-byte rows, 8-row groups 1024 B apart;
                            //    the k-th 16-wide slice starts 32 bytes further.
                            const uint64_t a_desc =
                                ptx::smem_desc_sw128(a_base + q * Cfg::A_SUB_BYTES + kk * 32, 16, 1024);
                            // B row-major: N-major, 64-column boxes B_ATOM_BYTES apart
                            //    (leading offset), 8 K-rows of 128 B per group (stride
                            //    offset); the k-th 16-row slice starts 16 * 128 bytes
                            //    further. B column-major: K-major like A.
                            // A narrow last part (32 or 16 columns per CTA): rows of
                            //    64 or 32 bytes in the swizzle of that width, 8
                            //    K-rows per group, the k-th 16-row slice 16 rows
                            //    further.
                            constexpr int TAIL_ROW = Cfg::TAIL_N;   // bytes per K-row of a CTA's tail box
                            const uint64_t b_desc =
                                Cfg::B_KMAJOR ? ptx::smem_desc_sw128(b_q + kk * 32, 16, 1024)
                                : (Cfg::NARROW_TAIL && part_cols == Cfg::TAIL_N)
                                    ? ptx::smem_desc(b_q + kk * 16 * TAIL_ROW, Cfg::B_TAIL_BYTES, 8 * TAIL_ROW,
                                                     TAIL_ROW == 64 ? ptx::kLayoutSw64 : ptx::kLayoutSw32)
                                    : ptx::smem_desc_sw128(b_q + kk * 2048, Cfg::B_ATOM_BYTES, 1024);
                            const bool acc = (kb != w.kb0) || k16 != skip16;
                            if constexpr (PAIR)
                                ptx::mma_f16_pair(d_part, a_desc, b_desc, idesc, acc);
                            else
                                ptx::mma_f16(d_part, a_desc, b_desc, idesc, acc);
                        }
                        pending = true;
                    }
                    if (!ok && !pending) break;
                    // (after a failed wait for part 1, part 0's MMAs still get
                    // their commit, so the drain below covers them)
                    issued = true;
                    if constexpr (PAIR)
                        ptx::mma_commit_pair_multicast(empty_bar(stage), 0x3);
                    else
                        ptx::mma_commit(empty_bar(stage));
                    if constexpr (Cfg::KSPLIT) {
                        // hand k-block g over: order this thread's MMAs so far
                        // before the arrive that the other thread waits on
                        ptx::tc_fence_before_sync();
                        ptx::mbar_arrive(handed_bar(stage));
                    }
                    next_stage();
                    if (!ok) break;
                }
                if (ok) {
                    if constexpr (PAIR)
                        ptx::mma_commit_pair_multicast(acc_full_bar(buf), 0x3);
                    else
                        ptx::mma_commit(acc_full_bar(buf));
                }
                walked += w.kb1 - w.kb0;
                ++local;
            }
            if (!ok && issued) {
                // Drain this thread's MMAs before tensor memory is released:
                // the last commit arrives on the stage before `stage`.
                const int last = (stage + STAGES - 1) % STAGES;
                waiter.drain(empty_bar(last), (stage == 0) ? (phase ^ 1u) : phase);
            }
        }
        __syncwarp();
    } else if (warp >= 2 && warp < 2 + Cfg::EPI_WARPS) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;             // tensor-memory lanes 32*quarter ..
        const int col_half = (warp - 2) / 4;      // with 8 warps: which half of each part's columns
        constexpr int COL_SPLIT = Cfg::EPI_WARPS / 4;
        const uint32_t buf_s = base + Cfg::OFF_EPI + static_cast<uint32_t>((warp - 2) * Cfg::EPI_CHUNK_BYTES);
        const bool read_c = (p.beta != 0.0f) && p.k_splits <= 1;
        int32_t local = 0;
        for (int32_t i = first_item; i < p.items; i += item_step) {
            const WorkItem w = work_item<BN, Cfg::STREAM_K>(p, i);
            if (w.n0 >= p.N) continue;
            int32_t cls, j0;
            a_class_of<Cfg::TILE_M, Cfg::A_CLASSES>(p, w.mb, cls, j0);
            const int32_t jb = j0 + static_cast<int32_t>(rank) * BM + quarter * 32;  // class row
            const int32_t rows = min(32, a_rows_of<Cfg::A_CLASSES>(p, cls) - jb);
            // C rows of class cls are cls, cls + P, cls + 2P, ...
            const int64_t row_stride = static_cast<int64_t>(p.a_classes) * p.ldc;
            float* c_tile = p.C + (cls + static_cast<int64_t>(p.a_classes) * jb) * p.ldc;
            const int32_t n0 = w.n0;
            const int accb = local % ACC_BUFS;
            const uint32_t acc_phase = (local / ACC_BUFS) & 1;
            // (stream-K: the tile's first k-blocks add onto C without reading it)
            const int32_t sk = Cfg::STREAM_K ? w.sk : kSkWhole;
            const bool item_read_c = read_c && sk != kSkFirst;
            // beta * C needs C's old values: this warp's rows of the item's C
            // are brought into L2 and the first chunk's loads go out now,
            // while the MMAs of this tile are still running (one bulk
            // prefetch per row and lane; the two warps of a lane quarter take
            // half of the item's columns each, widened to the 16-byte blocks
            // that hold the first and last elements)
            if (item_read_c && lane < rows) {
                const int32_t cend = min(n0 + w.width, p.N);
                const int32_t half = (cend - n0 + 1) / 2;
                const int32_t cb = n0 + col_half * half;
                const int32_t ce = min(cb + half, cend);
                if (ce > cb) {
                    const float* c_row = c_tile + static_cast<int64_t>(lane) * row_stride;
                    const uint64_t a = reinterpret_cast<uint64_t>(c_row + cb) & ~uint64_t{15};
                    const uint64_t e = (reinterpret_cast<uint64_t>(c_row + ce) + 15) & ~uint64_t{15};
                    ptx::bulk_prefetch_l2(a, static_cast<uint32_t>(e - a));
                }
            }
            float c_cur[32];
            if (item_read_c) {
                // (this warp's first columns of the first part handed back)
                const AccPart g0 = acc_part<Cfg>(0, accb, w.width);
                const int32_t col0 = n0 + g0.out_col + col_half * (g0.width / COL_SPLIT);
                if constexpr (Cfg::EPI_COLS == 16)
                    load_c_chunk16(c_tile, row_stride, col0, lane, p.N, rows, c_cur);
                else
                    load_c_chunk(c_tile, row_stride, col0 + lane, p.N, rows, c_cur);
            }
            if constexpr (Cfg::CSPLIT) {
                // the old C of this CTA's rows of the tile into L2 while the
                // slices run (one bulk prefetch per row)
                if (p.beta != 0.0f) {
                    const CsplitShare sh = csplit_share<Cfg>(p);
                    const int32_t r = sh.r0 + (warp - 2) * 32 + lane;
                    const int32_t cend = min(sh.n0 + BN, p.N);
                    if (r < sh.r1 && cend > sh.n0) {
                        const float* c_row = sh.c_tile + static_cast<int64_t>(r) * sh.row_stride;
                        const uint64_t a = reinterpret_cast<uint64_t>(c_row + sh.n0) & ~uint64_t{15};
                        const uint64_t e = (reinterpret_cast<uint64_t>(c_row + cend) + 15) & ~uint64_t{15};
                        ptx::bulk_prefetch_l2(a, static_cast<uint32_t>(e - a));
                    }
                }
            }
            const bool ready = waiter.wait(acc_full_bar(accb), acc_phase);
            if (!__all_sync(0xffffffffu, ready)) {
                if (lane == 0) waiter.fail(kRoleEpilogue, i);
                break;
            }
            ptx::tc_fence_after_sync();
            // Stream-K: wait until the warp holding the same rows and columns
            // in the next range has written them and published this call's
            // epoch in its flag
            if (sk == kSkFirst) {
                const int32_t* flag = p.sk_flags + ((w.range + 1) * Cfg::CTAS + static_cast<int32_t>(rank)) *
                                                       Cfg::EPI_WARPS + (warp - 2);
                bool got = ptx::ld_acquire_gpu(flag) == p.sk_epoch;
                if (!got) {
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (!(got = ptx::ld_acquire_gpu(flag) == p.sk_epoch) && !*abort_flag &&
                           ptx::globaltimer_ns() - t0 <= p.wait_limit_ns) {
                    }
                }
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) waiter.fail(kRoleEpilogue, i);
                    break;
                }
            }
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            if constexpr (Cfg::CSPLIT) {
                // this warp's 32 rows and half of the columns of the slice's
                // accumulator, unscaled, to the partial over the ring (the
                // tensor core has read the ring for the last time: the
                // accumulator is full)
                ptx::fence_proxy_async_smem();
                const int32_t row = quarter * 32 + lane;
#pragma unroll 1
                for (int32_t c = col_half * (BN / COL_SPLIT); c < (col_half + 1) * (BN / COL_SPLIT); c += 32) {
                    uint32_t r[32];
                    ptx::tmem_load_32x32b_x32(t_row + static_cast<uint32_t>(accb * BN + c), r);
                    ptx::tmem_load_wait();
                    ptx::tmem_regs_ready(r);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        ptx::st_shared_v4(base + Cfg::OFF_A + partial_off(row, c + 4 * q), __uint_as_float(r[4 * q]),
                                          __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                                          __uint_as_float(r[4 * q + 3]));
                }
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acc_empty_bar(accb, 0));
            } else {
            // the accumulator's parts in order (one part: the whole item);
            // each part goes back to the MMA warp as soon as it has been read,
            // and parts past the item's width are handed back at once
            for (int h = 0; h < RELEASE_PARTS; ++h) {
                const AccPart g = acc_part<Cfg>(h, accb, w.width);
                const int32_t my_n = g.width / COL_SPLIT;   // columns of the part this warp stores
                const int32_t my_off = col_half * my_n;
                const int32_t pn0 = n0 + g.out_col + my_off;
                // hand part h of the accumulator back to its MMA thread
                auto release = [&]() {
                    ptx::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            ptx::mbar_arrive_cluster(ptx::mapa_shared(acc_empty_bar(accb, h), 0));
                        else
                            ptx::mbar_arrive(acc_empty_bar(accb, h));
                    }
                };
                if (g.out_col < w.width) {
                    // this warp's columns of the part, within the item
                    const int32_t my_w = min(my_n, w.width - g.out_col - my_off);
                    if constexpr (Cfg::EPI_COLS == 16) {
                        if (h > 0 && item_read_c && my_w > 0)
                            load_c_chunk16(c_tile, row_stride, pn0, lane, p.N, rows, c_cur);
                        store_tile16<Cfg::STREAM_K>(p, &maps.c, t_row + static_cast<uint32_t>(g.tmem_col + my_off),
                                                    c_tile, row_stride, rows, jb, pn0, my_w, buf_s, lane, c_cur, sk,
                                                    release);
                    } else {
                        if (h > 0 && item_read_c && my_w > 0)
                            load_c_chunk(c_tile, row_stride, pn0 + lane, p.N, rows, c_cur);
                        store_tile<Cfg::STREAM_K, Cfg::EPI_BATCH_LOADS>(p, &maps.c, t_row + static_cast<uint32_t>(g.tmem_col + my_off), c_tile, row_stride,
                                   rows, jb, pn0, my_w, buf_s, lane, c_cur, sk, release);
                    }
                } else {
                    release();
                }
            }
            if (sk == kSkRest) {
                // every lane's stores of C visible at GPU scope before the flag
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    ptx::st_release_gpu(
                        p.sk_flags + (w.range * Cfg::CTAS + static_cast<int32_t>(rank)) * Cfg::EPI_WARPS + (warp - 2),
                        p.sk_epoch);
            }
            }   // (not CSPLIT)
            ++local;
        }
        // the TMA stores must have read this CTA's shared memory before the
        // CTA exits (their global writes complete with the kernel)
        if (p.c_tma && lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if constexpr (Cfg::CSPLIT) {
        // every slice's partial written; then this CTA's rows of the tile
        // summed over the cluster's partials, and the peers' reads of this
        // CTA's partial finished before it exits
        ptx::cluster_sync();
        csplit_reduce<Cfg>(p, base + Cfg::OFF_A);
        ptx::cluster_sync();
    }
    if constexpr (PAIR) {
        // After an abort the peer's loads into this pair may still be landing:
        // give them a moment before the cluster (and its shared memory) goes away.
        if (*abort_flag) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (ptx::globaltimer_ns() - t0 < 200000ull) {
            }
        }
        ptx::cluster_sync();
    }
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else
            ptx::tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace mpgemm
