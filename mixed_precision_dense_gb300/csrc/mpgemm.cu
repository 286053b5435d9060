// mpgemm: host side of the C ABI declared in include/mpgemm.h.
//
// mpgemm_run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream):
//   1. validate and classify (host): quick returns for M*N == 0 (nothing)
//      and K == 0 or alpha == 0 (C = beta*C); for A and B, whether base
//      address and row pitch are both multiples of 16 bytes, which the
//      tensor memory accelerator (TMA) requires;
//   2. stage an operand that fails that test into an aligned copy in the
//      handle's workspace (stage_rows_u16);
//   3. encode 2-D tensor maps with 128-byte swizzle and zero fill past the
//      matrix edge;
//   4. launch the persistent tensor-core kernel (gemm_kernel.cuh) with one
//      CTA per SM on `stream`.
// Everything is stream-ordered; nothing here synchronises the device.
//
// The operation: "Day 80, Capstone 4: a tensor-core GEMM" ("Capability",
// "Minimal model"); the alpha/beta scaling of its matched cublasGemmEx
// baseline ("Compare like with like"); ragged edges by zero fill ("Faded
// practice", practice 3: zero is safe for a matrix product); unaligned
// leading dimensions ("Common failures": a misaligned address is a broken
// load promise) by an aligned staging copy, the GB300 counterpart of the
// padded operand of "GEMM kernels 1-7 + Tensor Cores" (TC-02, K padded to
// 1008).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <algorithm>
#include <functional>
#include <numeric>
#include <mutex>
#include <vector>

#include "../../include/mpgemm.h"
#include "gemm_kernel.cuh"
#include "peak_probe.cuh"

namespace mpgemm {
namespace {

constexpr int64_t kDimLimit = (int64_t{1} << 31) - 1;
constexpr uint64_t kDefaultWaitLimitNs = 4000000000ull;

using Cfg256 = TileConfig<256, 4, false>;   // one CTA per 128 x 256 tile
using Cfg128 = TileConfig<128, 6, false>;   // one CTA per 128 x 128 tile
// one CTA per 128 x 320 tile (N from 257 to 320 in one tile column): 56 KB
// stages, so three of them, and one accumulator buffer
using Cfg320 = TileConfig<320, 3, false>;
using CfgPair = TileConfig<256, 3, true, false, 2, 2>;   // a CTA pair per 256 x 256 tile, two MMA issuers
                                                      // taking alternate k-blocks in a fixed order
using CfgWide = TileConfig<512, 4, true>;   // a CTA pair per 256 x 512 tile
// a CTA pair per 256 x 384 tile (parts of 256 and 128 columns, one MMA
// thread each; N from 257 to 384 in one tile column)
using CfgPair384 = TileConfig<384, 4, true, false, 2>;
// a CTA pair per 256 x 320 tile: parts of 256 and 64 columns, the 64-column
// part read in 32-column boxes per CTA (4 KB, 64-byte swizzle), so five 36 KB
// stages fit (N from 289 to 320, row-major B)
using CfgPair320 = TileConfig<320, 5, true, false, 2>;
// a CTA pair per 256 x 288 tile: parts of 256 and 32 columns, the 32-column
// part read in 16-column boxes per CTA (2 KB, 32-byte swizzle) (N from 257
// to 288, row-major B). With A in row classes, five 34 KB stages; with A
// read as it is (aligned or staged), three 68 KB stages of two k-blocks and
// 16-column epilogue chunks (2 KB buffers). Measured on GB300, L2 flushed,
// us, five stages of one k-block / three of two: 65536 x 257 x 4093 (lda
// 4093, 64 row classes) 163.8 / 164.2 at beta 0.5, 151.1 / 153.1 at beta 0;
// A aligned: 65536 x 280 x 4096, beta 0.5, 156.7 / 149.5; 65536 x 288 x
// 4096 133.5 / 129.2; 58368 x 264 x 4096 114.6 / 111.6. Before, 256 x 320
// pairs took 169.2 / 159.8 us on the first shape (A in 16-byte classes); a
// variant of three stages of two k-blocks whose eight epilogue warps shared
// four 32-column buffers (wrong results, an upper bound) took 160.5 / 147.3.
using CfgPair288 = TileConfig<288, 5, true, false, 2>;
using CfgPair288A = TileConfig<288, 3, true, false, 2, 2>;
// the same five shapes for a column-major B (a K-major B operand)
using Cfg256K = TileConfig<256, 4, false, true>;
using Cfg128K = TileConfig<128, 6, false, true>;
using Cfg320K = TileConfig<320, 3, false, true>;
using CfgPairK = TileConfig<256, 6, true, true, 2>;
using CfgWideK = TileConfig<512, 4, true, true>;
using CfgPair384K = TileConfig<384, 4, true, true, 2>;
// one-CTA 128 x 128 tiles whose K slices run as one cluster per tile and are
// summed through distributed shared memory (split-K in clusters)
using Cfg128C = TileConfig<128, 6, false, false, 1, 1, true>;
using Cfg128KC = TileConfig<128, 6, false, true, 1, 1, true>;
// largest cluster (slices per tile) the cluster split-K launches
constexpr int kMaxClusterSplits = kMaxClusterSlices;
// stream-K flags per range: one per CTA of the pair and epilogue warp
constexpr int kSkFlagsPerRange = 2 * CfgPair::EPI_WARPS;
static_assert(CfgPair::STREAM_K && CfgPair288::STREAM_K && CfgPair288A::STREAM_K && CfgPair320::STREAM_K &&
                  CfgPair384::STREAM_K && !CfgWide::STREAM_K && CfgPair288::EPI_WARPS == CfgPair::EPI_WARPS &&
                  CfgPair288A::EPI_WARPS == CfgPair::EPI_WARPS &&
                  CfgPair320::EPI_WARPS == CfgPair::EPI_WARPS && CfgPair384::EPI_WARPS == CfgPair::EPI_WARPS,
              "stream-K shapes");
// the kernels whose parameters hold 64 row classes of A (the rest hold 8)
static_assert(CfgPair288::A_CLASSES == kMaxAClasses && CfgPair320::A_CLASSES == kMaxAClasses &&
                  CfgPair288A::A_CLASSES == kTableAClasses &&
                  CfgPair384::A_CLASSES == kTableAClasses && CfgPair::A_CLASSES == kTableAClasses &&
                  CfgWide::A_CLASSES == kTableAClasses && Cfg320::A_CLASSES == kTableAClasses,
              "row-class capacities");
// one occupancy query (max_pair_clusters) serves both pair shapes: shared
// memory limits either to one CTA per SM, and both stay far below the SM's
// thread and register limits at that occupancy
static_assert(CfgWide::SMEM_BYTES > 232448 / 2 && CfgPair::SMEM_BYTES > 232448 / 2 &&
                  CfgPair384::SMEM_BYTES > 232448 / 2 && CfgPair320::SMEM_BYTES > 232448 / 2 &&
                  CfgPair288::SMEM_BYTES > 232448 / 2 && CfgPair288A::SMEM_BYTES > 232448 / 2 &&
                  CfgWide::THREADS <= 384 && CfgPair::THREADS <= 384 && CfgPair384::THREADS <= 384 &&
                  CfgPair320::THREADS <= 384 && CfgPair288::THREADS <= 384 && CfgPair288A::THREADS <= 384,
              "the wide pair kernel fits wherever the 256 x 256 pair kernel fits");

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

struct Options {
    int32_t b_col_major = 0;        // per call: B(k, j) = B[j*ldb + k]
    int32_t tile_m = 0;
    int32_t tile_n = 0;
    int32_t max_ctas = 0;
    int32_t force_staging = 0;
    int32_t raster_group = 0;
    int32_t l2_keep = 0;            // 0 automatic, 1 keep A, 2 keep B
    int32_t split_k = 0;            // 0 automatic, 1 never, n >= 2: n slices of K per tile
    int32_t pair_units = 0;         // CTA pairs resident at once (0: num_sms / 2)
    int32_t test_stall = 0;
    int32_t c_store = 0;            // 0 automatic (TMA stores when possible), 1 per-lane stores
    int32_t acc16 = 0;              // 1: FP16 accumulators (study variant)
    int32_t reproducible = 0;       // 1: only paths whose summation order is fixed
    int32_t stream_k = 0;           // 0 automatic, 1 never, 2 whenever the tile shape allows
    int32_t split_reduce = 0;       // 0 automatic (clusters for reproducible calls), 1 atomics /
                                    // reduce-adds, 2 clusters where possible
    uint64_t wait_limit_ns = kDefaultWaitLimitNs;
};

bool aligned16(const void* p, int64_t ld_elems, int64_t elem_bytes) {
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld_elems * elem_bytes) % 16 == 0);
}

mpgemm_status_t validate(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                         const void* B, int64_t ldb, float beta, const void* C, int64_t ldc,
                         int32_t b_col_major = 0) {
    const int64_t b_min = b_col_major ? K : N;   // row length of B as stored
    if (M < 0 || N < 0 || K < 0) return MPGEMM_ERR_INVALID_VALUE;
    if (M > kDimLimit || N > kDimLimit || K > kDimLimit) return MPGEMM_ERR_INVALID_VALUE;
    if (lda < (K > 1 ? K : 1) || ldb < (b_min > 1 ? b_min : 1) || ldc < (N > 1 ? N : 1))
        return MPGEMM_ERR_INVALID_VALUE;
    if (lda > kDimLimit || ldb > kDimLimit || ldc > kDimLimit) return MPGEMM_ERR_INVALID_VALUE;
    if (M > 0 && N > 0 && K > 0 && M * N > (int64_t{1} << 62) / K) return MPGEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return MPGEMM_OK;
    if (!C || reinterpret_cast<uintptr_t>(C) % 4 != 0) return MPGEMM_ERR_INVALID_VALUE;
    if (K > 0 && alpha != 0.0f) {
        if (!A || !B) return MPGEMM_ERR_INVALID_VALUE;
        if (reinterpret_cast<uintptr_t>(A) % 2 != 0 || reinterpret_cast<uintptr_t>(B) % 2 != 0)
            return MPGEMM_ERR_INVALID_VALUE;
    }
    (void)beta;
    return MPGEMM_OK;
}

// 256-wide tiles move less operand data per FLOP; they are worth it as soon
// as they keep at least four fifths of the SMs busy.
//
// When N is 257 to 320, 256-wide tiles leave a second tile column of at most
// 64 columns, whose tiles read all of A again. One 320-wide tile column
// reads A once, but its 56 KB stages leave room for three, and at these
// shapes a k-block takes about the load latency over the stages in flight,
// whatever their size: a wave of 320-wide tiles costs 1.9 waves of 256-wide
// ones when A is aligned, 1.6 when A is read in row classes (each read of an
// unaligned row touches an extra cache line, and the 256-wide walk reads
// every row twice). Measured on GB300 at N = 257, K = 4093, beta = 0.5, in
// us per call, 256 -> 320 wide: M = 58368 (three waves of 320-wide tiles)
// 181.5 -> 168.6 aligned, 229.6 -> 179.9 in row classes; M = 65536 (3.4
// waves) 202.2 -> 221.0 and 257.5 -> 225.2; M = 77824 (four waves) 231.8 ->
// 224.3 and 287.8 -> 237.7. The choice compares whole waves.
int32_t auto_tile_n(int64_t M, int64_t N, int32_t num_sms, bool a_row_classes) {
    if (N <= 128) return 128;
    const int64_t m_tiles = ceil_div(M, 128);
    const int64_t tiles256 = m_tiles * ceil_div(N, 256);
    const bool wide = tiles256 * 5 >= static_cast<int64_t>(num_sms) * 4;
    if (wide && N > 256 && N <= 320) {
        const double wave320 = a_row_classes ? 1.6 : 1.9;   // in waves of 256-wide tiles
        if (static_cast<double>(ceil_div(m_tiles, num_sms)) * wave320 <
            static_cast<double>(ceil_div(tiles256, num_sms)))
            return 320;
    }
    return wide ? 256 : 128;
}

// N from 257 to 384 in one tile column of CTA pairs (256 x 320 tiles, or
// 256 x 384 past 320 columns or for a column-major B) once those tiles fill
// every pair: A is read once, and each SM receives half of B per k-block.
// Measured on GB300 at 65536 x 257 x 4093 (lda 4093, beta = 0.5): 182 us in
// 256 x 320 pairs, 185 us in 256 x 384 pairs, 218 us in one-CTA 128 x 320
// tiles; with A aligned at 58368 rows, 135 against 169 us.
bool auto_narrow_pair(int64_t M, int64_t N, int32_t num_sms) {
    return N > 256 && N <= 384 && ceil_div(M, 256) >= num_sms / 2;
}

// CTA pairs (256 x 256 tiles) pay off once there is at least a full wave of
// pair tiles and the last column band wastes at most a fifth of its width;
// with a long K (3072 or more), also when the pair tiles keep four fifths
// of the pairs busy (their operand feed per SM is two thirds of a 128 x 256
// CTA's: 2048 x 2048 x 4096 ran 7 % faster in 64 pair tiles than in 128
// one-CTA tiles, 2048^3 equally fast).
bool auto_pair(int64_t M, int64_t N, int64_t K, int32_t num_sms) {
    if (M < 512 || N < 512) return false;
    if (ceil_div(N, 256) * 256 * 4 > 5 * N) return false;
    const int64_t tiles = ceil_div(M, 256) * ceil_div(N, 256), units = num_sms / 2;
    return tiles >= units || (K >= 3072 && tiles * 5 >= units * 4);
}

// Time of a persistent walk over `tiles` tiles on `units` CTA pairs, in
// tile times: full waves, plus half a wave when the last wave is at most half
// full (its tiles then run as half-width items), else a whole wave.
double pair_waves(int64_t tiles, int64_t units) {
    const int64_t full = tiles / units, rem = tiles % units;
    return static_cast<double>(full) + (rem == 0 ? 0.0 : (2 * rem <= units && full > 0 ? 0.5 : 1.0));
}

// Pair tiles 512 wide instead of 256: each SM then receives 48 KB of operands
// per 1024 MMA cycles instead of 32 KB per 512; the price is a single
// accumulator buffer, whose epilogue overlaps the next tile only by halves,
// and coarser waves. The relative efficiencies within a tile weigh the two
// walks against each other (measured at the power cap, cycles per launch
// corrected for the waves: 1.085 at 8192^3, 1.12 at 6144^3, 1.02 at
// 16384 x 16384 x 4096); below K = 2048 the exposed epilogue is no longer
// paid for.
bool auto_wide(int64_t M, int64_t N, int64_t K, int64_t units) {
    if (K < 2048 || N < 1024) return false;
    constexpr double kEff256 = 0.83, kEff512 = 0.83 * 1.07;
    const int64_t mt = ceil_div(M, 256);
    const double t256 = pair_waves(mt * ceil_div(N, 256), units) / kEff256;
    const double t512 = 2.0 * pair_waves(mt * ceil_div(N, 512), units) / kEff512;
    return t512 < t256;
}

// How the tensor-core pass reads A (see kMaxAClasses in gemm_kernel.cuh): one
// row class when A's rows start on 16-byte boundaries (or A was staged), else
// P classes of rows i = r (mod P), each read from the U-aligned address at or
// below row r with a shift of (address mod U) / 2 elements, where U = 128
// when P * lda * 2 is a multiple of 128 (every row of a class then starts at
// the same offset in its L2 line, and every box row of A is one whole line),
// else 16. The planner takes P = 16 / gcd(2 lda, 16), or P = 128 / gcd(2 lda,
// 128) (up to 64) when the kernel has room for that many classes and they
// cost at most 1/32 more tiles.
int32_t a_class_unit(int64_t P, int64_t lda) { return (P * 2 * lda) % 128 == 0 ? 128 : 16; }

int64_t a_class_tiles(int64_t M, int64_t P, int64_t tile_m) {
    int64_t tiles = 0;
    for (int64_t r = 0; r < P && r < M; ++r) tiles += ceil_div((M - r + P - 1) / P, tile_m);
    return tiles;
}

int32_t choose_a_classes(int64_t lda, int64_t M, int64_t tile_m, int32_t capacity) {
    const int64_t p16 = 16 / std::gcd<int64_t>(2 * lda, 16);
    const int64_t p128 = 128 / std::gcd<int64_t>(2 * lda, 128);
    if (p128 > p16 && p128 <= capacity &&
        a_class_tiles(M, p128, tile_m) * 32 <= a_class_tiles(M, p16, tile_m) * 33)
        return static_cast<int32_t>(p128);
    return static_cast<int32_t>(p16);
}

struct AClassLayout {
    int32_t P = 1;
    int32_t unit = 16;   // U
    int32_t max_shift = 0;
    int32_t shift[kMaxAClasses] = {};
    int64_t rows[kMaxAClasses] = {};
    int64_t first_tile[kMaxAClasses + 1] = {};
    uintptr_t base[kMaxAClasses] = {};
};

// classes: the P chosen by the planner, or 0 (one class, no shift)
AClassLayout a_class_layout(const void* A, int64_t lda, int64_t M, int32_t classes, int64_t tile_m) {
    AClassLayout L;
    const uintptr_t a = reinterpret_cast<uintptr_t>(A);
    L.P = classes > 0 ? std::min(classes, kMaxAClasses) : 1;
    L.unit = classes > 0 ? a_class_unit(L.P, lda) : 16;
    for (int32_t r = 0; r < L.P; ++r) {
        const uintptr_t addr = a + static_cast<uintptr_t>(r) * static_cast<uintptr_t>(lda) * 2;
        const int32_t off = classes > 0 ? static_cast<int32_t>(addr % static_cast<uintptr_t>(L.unit)) : 0;
        L.shift[r] = off / 2;
        L.max_shift = std::max(L.max_shift, L.shift[r]);
        L.base[r] = addr - off;
        L.rows[r] = r < M ? (M - r + L.P - 1) / L.P : 0;
        L.first_tile[r + 1] = L.first_tile[r] + ceil_div(L.rows[r], tile_m);
    }
    return L;
}

// The stream-K ranges: range r is [start[r], start[r + 1]) of the tiles'
// k-blocks (units = tiles * k_blocks), R ranges of about equal length. A
// boundary that would leave a piece of a tile of an eighth of its k-blocks
// or fewer on either side moves to the tile's edge: such a piece costs a
// whole epilogue (and, inside a range, stalls the next tile's MMAs behind
// the drain) for a few k-blocks of work. Without the moves when they would
// leave a range shorter than one tile's k-blocks. Measured on GB300, L2
// flushed, us, equal ranges / moved / ranges balanced on k-blocks plus a
// cost per tile touched (eighth or quarter of a tile):
//   65536 x 257 x 4093, beta 0.5: 171.4 / 169.2 / 169.9, 167.6
//   65536 x 257 x 4093, beta 0:   158.5 / 158.6 / 167.7, 167.4
//   65536 x 300 x 4096, beta 0:   -     / 140.8 / 150.9, 150.4
std::vector<int32_t> sk_range_starts(int64_t units, int64_t k_blocks, int64_t R) {
    std::vector<int32_t> start(static_cast<size_t>(R + 1));
    const int64_t len = units / R, rem = units % R, snap = std::max<int64_t>(1, k_blocks / 8);
    for (int64_t r = 0; r <= R; ++r) start[r] = static_cast<int32_t>(r * len + std::min(r, rem));
    std::vector<int32_t> moved = start;
    for (int64_t r = 1; r < R; ++r) {
        const int64_t off = moved[r] % k_blocks;
        if (off != 0 && off <= snap)
            moved[r] = static_cast<int32_t>(moved[r] - off);
        else if (off != 0 && k_blocks - off <= snap)
            moved[r] = static_cast<int32_t>(moved[r] + (k_blocks - off));
    }
    for (int64_t r = 0; r < R; ++r)
        if (moved[r + 1] - moved[r] < k_blocks) return start;
    return moved;
}

// 64-wide k-blocks per pipeline stage of the kernel a plan launches (the
// 256 x 288 pair: two for an A read as it is, one for A in row classes).
int32_t plan_kps(int32_t tile_m, int32_t tile_n, bool b_col_major, bool a_classes = false) {
    if (tile_m == 256) {
        if (tile_n == 512) return b_col_major ? CfgWideK::KPS : CfgWide::KPS;
        if (tile_n == 384) return b_col_major ? CfgPair384K::KPS : CfgPair384::KPS;
        if (tile_n == 320) return CfgPair320::KPS;
        if (tile_n == 288) return a_classes ? CfgPair288::KPS : CfgPair288A::KPS;
        return b_col_major ? CfgPairK::KPS : CfgPair::KPS;
    }
    if (tile_n == 320) return b_col_major ? Cfg320K::KPS : Cfg320::KPS;
    if (tile_n == 256) return b_col_major ? Cfg256K::KPS : Cfg256::KPS;
    return b_col_major ? Cfg128K::KPS : Cfg128::KPS;
}

mpgemm_status_t make_plan(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                          const void* B, int64_t ldb, float beta, const void* C, int64_t ldc,
                          int32_t num_sms, const Options& opt, mpgemm_plan_t* out) {
    mpgemm_status_t st = validate(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, opt.b_col_major);
    if (st != MPGEMM_OK) return st;
    if (num_sms <= 0) return MPGEMM_ERR_INVALID_VALUE;
    if (opt.tile_n == 512 && opt.tile_m == 128) return MPGEMM_ERR_INVALID_VALUE;   // 512 wide: pairs only
    // 256 x 320 and 256 x 288 pairs read B in narrow row-major boxes; 288 wide: pairs only
    if (opt.tile_n == 320 && opt.tile_m == 256 && opt.b_col_major) return MPGEMM_ERR_INVALID_VALUE;
    if (opt.tile_n == 288 && (opt.tile_m == 128 || opt.b_col_major)) return MPGEMM_ERR_INVALID_VALUE;
    if (opt.tile_n == 384 && opt.tile_m == 128) return MPGEMM_ERR_INVALID_VALUE;   // 384 wide: pairs only
    mpgemm_plan_t p;
    std::memset(&p, 0, sizeof(p));
    p.tile_m = 128;
    p.tile_k = 64;
    if (M == 0 || N == 0) {
        p.quick = 1;
    } else if (K == 0 || alpha == 0.0f) {
        p.quick = 2;
    }
    if (p.quick) {
        *out = p;
        return MPGEMM_OK;
    }
    p.stage_b = (opt.force_staging || !aligned16(B, ldb, 2)) ? 1 : 0;
    const bool narrow_pair = !opt.tile_m && !opt.tile_n && auto_narrow_pair(M, N, num_sms);
    const bool pair = opt.tile_n == 512 || opt.tile_n == 384 || opt.tile_n == 288 || narrow_pair ||
                      (opt.tile_m ? (opt.tile_m == 256) : (!opt.tile_n && auto_pair(M, N, K, num_sms)));
    if (pair) {
        int64_t pair_units = num_sms / 2;
        if (opt.pair_units > 0) pair_units = std::min<int64_t>(pair_units, opt.pair_units);
        if (opt.max_ctas > 0) pair_units = std::min<int64_t>(pair_units, std::max<int64_t>(1, opt.max_ctas / 2));
        pair_units = std::max<int64_t>(1, pair_units);
        const bool wide = opt.tile_n == 512 || (!opt.tile_m && !opt.tile_n && auto_wide(M, N, K, pair_units));
        p.tile_m = 256;
        p.tile_n = (opt.tile_n == 384 || opt.tile_n == 320 || opt.tile_n == 288) ? opt.tile_n : (wide ? 512 : 256);
        if (narrow_pair) p.tile_n = opt.b_col_major ? 384 : N <= 288 ? 288 : N <= 320 ? 320 : 384;
        p.stages = p.tile_n == 384   ? CfgPair384::STAGES
                   : p.tile_n == 320 ? CfgPair320::STAGES
                   : p.tile_n == 288 ? CfgPair288::STAGES
                                     : (wide ? CfgWide::STAGES : CfgPair::STAGES);
        p.smem_bytes = p.tile_n == 384   ? CfgPair384::SMEM_BYTES
                       : p.tile_n == 320 ? CfgPair320::SMEM_BYTES
                       : p.tile_n == 288 ? CfgPair288::SMEM_BYTES
                                         : (wide ? CfgWide::SMEM_BYTES : CfgPair::SMEM_BYTES);
    } else {
        // (A is read in row classes below when its rows break the 16-byte rule)
        const bool row_classes = !aligned16(A, lda, 2) && !opt.force_staging && !opt.b_col_major;
        p.tile_n = opt.tile_n ? opt.tile_n : auto_tile_n(M, N, num_sms, row_classes);
        p.stages = p.tile_n == 320 ? Cfg320::STAGES : (p.tile_n == 256) ? Cfg256::STAGES : Cfg128::STAGES;
        p.smem_bytes = p.tile_n == 320   ? Cfg320::SMEM_BYTES
                       : p.tile_n == 256 ? Cfg256::SMEM_BYTES
                                         : Cfg128::SMEM_BYTES;
    }
    // An A whose rows break TMA's 16-byte rule is read in row classes
    // (row-major B), else copied to an aligned buffer.
    const bool a_aligned = aligned16(A, lda, 2);
    const bool a_classes = !a_aligned && !opt.force_staging && !opt.b_col_major;
    p.stage_a = (opt.force_staging || (!a_aligned && !a_classes)) ? 1 : 0;
    // room for 64 classes in the row-major pairs of 288 and 320 columns
    const int32_t class_room = (pair && !opt.b_col_major && (p.tile_n == 288 || p.tile_n == 320))
                                   ? CfgPair320::A_CLASSES
                                   : kTableAClasses;
    p.a_classes = a_classes ? choose_a_classes(lda, M, p.tile_m, class_room) : 0;
    const AClassLayout L = a_class_layout(A, lda, M, p.a_classes, p.tile_m);
    const int64_t m_tiles = L.first_tile[L.P], n_tiles = ceil_div(N, p.tile_n);
    p.tile_k = 64 * plan_kps(p.tile_m, p.tile_n, opt.b_col_major != 0, p.a_classes > 0);
    if (p.tile_m == 256 && p.tile_n == 288 && p.tile_k == 128) {   // A read as it is
        p.stages = CfgPair288A::STAGES;
        p.smem_bytes = CfgPair288A::SMEM_BYTES;
    }
    const int64_t k_blocks = ceil_div(K + L.max_shift, p.tile_k);
    if (m_tiles * n_tiles > kDimLimit / 2) return MPGEMM_ERR_INVALID_VALUE;
    p.m_tiles = static_cast<int32_t>(m_tiles);
    p.n_tiles = static_cast<int32_t>(n_tiles);
    p.k_blocks = static_cast<int32_t>(k_blocks);
    p.tiles = m_tiles * n_tiles;
    p.last_k_valid = static_cast<int32_t>(K - (k_blocks - 1) * p.tile_k);
    // persistent grid: one CTA (single) or one CTA pair (pair) per SM or SM pair
    const int64_t per_unit = pair ? 2 : 1;
    int64_t units = num_sms / per_unit;
    if (pair && opt.pair_units > 0) units = std::min<int64_t>(units, opt.pair_units);
    if (opt.max_ctas > 0) units = std::min<int64_t>(units, std::max<int64_t>(1, opt.max_ctas / per_unit));
    units = std::max<int64_t>(1, units);
    // Split-K (single-CTA tiles): when the tiles occupy at most a quarter of
    // the CTAs and K is long (32 k-blocks or more), cut each tile's K range
    // into slices of at least eight k-blocks; the slices' partial products are
    // added into C. Shorter problems lose more to the extra pass over C and
    // the atomic adds than they gain from the extra SMs. With beta == 1 the
    // slices add straight onto C and no pass over C is needed, so half of the
    // CTAs idle and 16 k-blocks already pay (1000 x 800 x 1200: 21 -> 17 us
    // with two slices). Very few tiles (an eighth of the SMs at most) pay
    // from eight k-blocks on (below).
    int64_t splits = 1;
    // (FP16 accumulators never split K: the study variant keeps the whole K
    // range in one FP16 accumulator, as an __half accumulator type would)
    if (!pair && opt.split_k != 1 && !opt.acc16) {
        if (opt.split_k >= 2)
            splits = opt.split_k;
        else if (beta == 1.0f ? (p.tiles * 2 <= units && k_blocks >= 16) : (p.tiles * 4 <= units && k_blocks >= 32))
            splits = std::min<int64_t>(k_blocks / 8, units / p.tiles);
        else if (p.tiles * 8 <= units && k_blocks >= 8)
            // very few tiles of a short K: five slices of two or more k-blocks
            // (measured with L2 flushed and beta != 1: 500 x 256 x 1024, 8
            // tiles, 12.3 -> 10.2 us; 300 x 200 x 640, 6 tiles, 10.7 -> 10.2
            // us; 200 x 136 x 617, 16 tiles, 12.5 -> 11.6 us; 40 tiles of 611 x
            // 613 x 617 slowed from 14.3 to 18-20 us, so not past an eighth of
            // the SMs). With beta == 1 the slices need no pass over C first,
            // so the split only costs less.
            splits = std::min<int64_t>(5, k_blocks / 2);
        splits = std::max<int64_t>(1, std::min<int64_t>(splits, k_blocks));
        if (splits > 1) splits = ceil_div(k_blocks, ceil_div(k_blocks, splits));  // no empty slice
    }
    // Split-K in clusters (MPGEMM_OPT_SPLIT_REDUCE): 128 x 128 tiles of at
    // most 8 slices, every slice of every tile resident at once (one CTA per
    // item): the slices of a tile run as one cluster and are summed through
    // distributed shared memory, in a fixed order, into one write of C.
    // Otherwise they add into C (after a pass applying beta), in the order
    // they finish, which a reproducible call does not allow. The clusters
    // cost 1.3-4 us more per call on GB300 (200 x 136 x 617: 11.1 -> 12.4;
    // 1000 x 800 x 1200, beta 1: 12.4 -> 16.5; 4096 x 16 x 4096: 16.1 ->
    // 18.7): their two cluster barriers and the partials' round trip
    // through shared memory are not hidden, where the slices' reduce-adds
    // run behind the next work. So they are the default only where the
    // order matters (reproducible calls), which then split K at all.
    const bool clusters = opt.split_reduce == 2 || (opt.split_reduce == 0 && opt.reproducible);
    if (splits > kMaxClusterSplits && clusters && p.tile_n == 128)
        splits = ceil_div(k_blocks, ceil_div(k_blocks, kMaxClusterSplits));
    p.split_reduce =
        (splits > 1 && clusters && p.tile_n == 128 && splits <= kMaxClusterSplits && p.tiles * splits <= units)
            ? 1
            : 0;
    if (splits > 1 && !p.split_reduce && opt.reproducible) splits = 1;
    p.k_splits = static_cast<int32_t>(splits);
    if (splits > 1) {
        p.split_tiles = 0;
        p.items = p.tiles * splits;
    } else {
        // If the last wave of tiles would keep at most half of the CTAs (pairs)
        // busy, do those tiles as two half-width items each: the wave then
        // finishes in half the time. (Not 288-, 320- or 384-wide tiles: a
        // half does not follow their 256 + 32, 256 + 64 or 256 + 128 column
        // parts.)
        const int64_t tile_units = std::min<int64_t>(units, p.tiles);
        const int64_t rem = p.tiles % tile_units;
        p.split_tiles = (p.tile_n != 288 && p.tile_n != 320 && p.tile_n != 384 && p.tiles > tile_units && rem > 0 &&
                         2 * rem <= tile_units)
                            ? static_cast<int32_t>(rem)
                            : 0;
        p.items = p.tiles + p.split_tiles;
    }
    // Stream-K (MPGEMM_OPT_STREAM_K): CTA pairs of 256 to 384 columns with at
    // least one tile per pair may walk one contiguous range of k-blocks each
    // instead of whole tiles. Automatic for tall-skinny problems (the 288-,
    // 320- and 384-wide pairs, or one column of 256-wide tiles) when the last wave
    // of tiles leaves pairs idle. Measured on GB300 with L2 flushed, us:
    //   65536 x 257 x 4093, beta 0.5 (256 tiles on 76 pairs): 186 -> 172;
    //   65536 x 256 x 4096: 121 -> 112 (beta 0), 135 -> 130 (beta 0.5);
    // and slower for square and wide problems on 256 x 256 pairs (6144^3:
    // 311 -> 361; 20480 x 1024 x 4096: 159 -> 171), whose cut tiles cost a
    // second pass over C while their pairs still drain whole tiles.
    p.sk_ranges = 0;
    if (pair && splits == 1 && !opt.acc16 && opt.stream_k != 1 && p.tile_n <= 384 && p.tiles >= units) {
        const int64_t sk_units = p.tiles * k_blocks;
        const bool want =
            opt.stream_k == 2 || ((p.tile_n > 256 || p.n_tiles == 1) && p.tiles % units != 0);
        if (want && sk_units < (int64_t{1} << 31) && units <= kMaxSkRanges) {
            p.sk_ranges = static_cast<int32_t>(units);
            p.split_tiles = 0;
            // items: every range walks as many as the range touching most tiles
            const std::vector<int32_t> start = sk_range_starts(sk_units, k_blocks, units);
            int64_t most = 1;
            for (int64_t r = 0; r < units; ++r)
                most = std::max<int64_t>(most, (start[r + 1] - 1) / k_blocks - start[r] / k_blocks + 1);
            p.items = units * most;
        }
    }
    if (p.items > kDimLimit) return MPGEMM_ERR_INVALID_VALUE;
    units = std::min<int64_t>(units, p.items);
    p.grid = static_cast<int32_t>(units * per_unit);
    int32_t group = opt.raster_group ? opt.raster_group : 16;
    if (group > p.m_tiles) group = p.m_tiles;
    p.raster_group = group;
    int64_t ws = 0;
    if (p.stage_a) ws += round_up(M * round_up(K, 8) * 2, 256);
    if (p.stage_b)
        ws += opt.b_col_major ? round_up(N * round_up(K, 8) * 2, 256) : round_up(K * round_up(N, 8) * 2, 256);
    p.workspace_bytes = ws;
    *out = p;
    return MPGEMM_OK;
}

// ------------------------------------------------------------------ kernels

// dst[r][c] = src[r][c] for c < cols, zero for cols <= c < round_up(cols, 8);
// 16-bit elements; dst rows are 16-byte aligned, src rows only 2-byte aligned.
// One thread per 16-byte output chunk: it reads the (one or two) aligned
// 16-byte source chunks that hold the chunk's eight elements and shifts them
// into place in registers. A source chunk is read only if it holds at least
// one element of the row, so no read leaves the 16-byte blocks the operand
// occupies.
__global__ void stage_rows_u16(const uint16_t* __restrict__ src, int64_t lds,
                               uint16_t* __restrict__ dst, int64_t ldd, int64_t rows,
                               int64_t cols) {
    const int64_t chunks = (cols + 7) / 8;
    const int64_t total = rows * chunks;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = idx / chunks;
        const int64_t c = (idx - r * chunks) * 8;
        const uintptr_t row_begin = reinterpret_cast<uintptr_t>(src + r * lds);
        const uintptr_t row_end = row_begin + 2 * static_cast<uintptr_t>(cols);
        const uintptr_t a = row_begin + 2 * static_cast<uintptr_t>(c);
        const uintptr_t a0 = a & ~static_cast<uintptr_t>(15);
        const uint32_t sh = static_cast<uint32_t>(a - a0);       // 0, 2, ..., 14
        uint32_t w[8];
        const uint4 lo = __ldg(reinterpret_cast<const uint4*>(a0));
        w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
        if (sh != 0 && a0 + 16 < row_end) {
            const uint4 hi = __ldg(reinterpret_cast<const uint4*>(a0 + 16));
            w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
        } else {
            w[4] = w[5] = w[6] = w[7] = 0u;
        }
        // words q .. q+4 of the 32 loaded bytes, q = sh / 4, without dynamic indexing
        const uint32_t q = sh >> 2;
        uint32_t v[5];
#pragma unroll
        for (int i = 0; i < 5; ++i)
            v[i] = q == 0 ? w[i] : (q == 1 ? w[i + 1] : (q == 2 ? w[i + 2] : w[i + 3]));
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = (sh & 2) ? __funnelshift_r(v[j], v[j + 1], 16) : v[j];
        const int64_t valid = cols - c;                           // >= 1
        if (valid < 8) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (2 * j >= valid) o[j] = 0u;
                else if (2 * j + 1 >= valid) o[j] &= 0xFFFFu;
            }
        }
        *reinterpret_cast<uint4*>(dst + r * ldd + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// C = beta * C over M x N (beta == 0 writes zeros without reading C).
// The GEMM launched after it (programmatic dependent launch) may start its
// loads and MMAs at once; its epilogue waits for this pass to complete.
__global__ void scale_c(float* __restrict__ C, int64_t ldc, int64_t M, int64_t N, float beta) {
    ptx::griddep_launch_dependents();
    const int64_t total = M * N;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = idx / N, j = idx - (idx / N) * N;
        float* p = C + i * ldc + j;
        *p = (beta == 0.0f) ? 0.0f : beta * *p;
    }
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Encoded tensor maps kept by a handle and reused by later calls with the
// same arguments. A map is a pure function of them (element type, base
// address, shape, pitch, box), so an entry never goes stale, even if the
// memory is freed and another buffer is placed at the same address; the least
// recently used entry is replaced. Host-side only: encoding costs a driver
// call per map per GEMM otherwise.
struct MapCache {
    static constexpr int kEntries = 16;
    struct Entry {
        uint64_t key[6];
        CUtensorMap map;
        uint64_t used;
        bool valid;
    };
    Entry e[kEntries] = {};
    uint64_t clock = 0;

    bool find(const uint64_t (&k)[6], CUtensorMap* out) {
        for (Entry& x : e) {
            if (x.valid && std::equal(k, k + 6, x.key)) {
                x.used = ++clock;
                *out = x.map;
                return true;
            }
        }
        return false;
    }
    void put(const uint64_t (&k)[6], const CUtensorMap& m) {
        Entry* victim = &e[0];
        for (Entry& x : e) {
            if (!x.valid) { victim = &x; break; }
            if (x.used < victim->used) victim = &x;
        }
        std::copy(k, k + 6, victim->key);
        victim->map = m;
        victim->used = ++clock;
        victim->valid = true;
    }

    // Whole sets of A's class maps when there are more classes than the
    // entries above hold (up to 64 for one call): keyed by the call's A
    // (address, pitch, rows, K, classes), two sets kept.
    struct ClassSet {
        uint64_t key[6];
        int32_t n;
        CUtensorMap a[kMaxAClasses];
        uint64_t used;
        bool valid;
    };
    ClassSet sets[2] = {};

    bool find_set(const uint64_t (&k)[6], CUtensorMap* out) {
        for (ClassSet& x : sets) {
            if (x.valid && std::equal(k, k + 6, x.key)) {
                x.used = ++clock;
                std::copy(x.a, x.a + x.n, out);
                return true;
            }
        }
        return false;
    }
    void put_set(const uint64_t (&k)[6], const CUtensorMap* a, int32_t n) {
        ClassSet* victim = !sets[0].valid ? &sets[0] : !sets[1].valid ? &sets[1]
                           : (sets[0].used <= sets[1].used ? &sets[0] : &sets[1]);
        std::copy(k, k + 6, victim->key);
        victim->n = n;
        std::copy(a, a + n, victim->a);
        victim->used = ++clock;
        victim->valid = true;
    }
};

// Row-major FP16 matrix rows x cols with pitch ld (elements), boxes of
// box_cols x box_rows, 128-byte swizzle (or `swizzle`), zeros outside the matrix, 128-byte
// L2 promotion (the box rows are 128 bytes; 256-byte promotion was 8 % slower
// on 65536 x 257 x 4093 and made no difference on square shapes).
bool encode_f16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                uint32_t box_cols, uint32_t box_rows, MapCache* cache = nullptr,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    const uint64_t key[6] = {16 | (static_cast<uint64_t>(swizzle) << 8), reinterpret_cast<uintptr_t>(base),
                             static_cast<uint64_t>(rows),
                             static_cast<uint64_t>(cols), static_cast<uint64_t>(ld),
                             (static_cast<uint64_t>(box_cols) << 32) | box_rows};
    if (cache && cache->find(key, map)) return true;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const bool ok = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    if (ok && cache) cache->put(key, *map);
    return ok;
}

int grid_for(int64_t work, int num_sms) {
    const int64_t blocks = ceil_div(work, 256);
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

template <class Cfg>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(gemm_tc_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::SMEM_BYTES);
}

// The kernel's tensor maps, cut down to the row classes it has room for
// (the planner never gives it more).
template <int NC>
TensorMapsT<NC> maps_for(const TensorMaps& ta) {
    if constexpr (NC == kMaxAClasses) {
        return ta;
    } else {
        TensorMapsT<NC> t;
        std::copy(ta.a, ta.a + NC, t.a);
        t.c = ta.c;
        t.b_tail = ta.b_tail;
        return t;
    }
}

template <class Cfg>
cudaError_t launch_tc(int grid, const TensorMaps& ta, const CUtensorMap& tb, const GemmParams& gp,
                      cudaStream_t stream) {
    if (gp.a_classes > Cfg::A_CLASSES) return cudaErrorInvalidValue;
    const TensorMapsT<Cfg::A_CLASSES> maps = maps_for<Cfg::A_CLASSES>(ta);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (Cfg::PAIR || Cfg::CSPLIT) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = Cfg::PAIR ? 2u : static_cast<unsigned>(gp.k_splits);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<Cfg>, maps, tb, gp);
}

// Clusters of two CTAs of the pair kernel that fit on the device at once.
int max_pair_clusters() {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(CfgPair::THREADS, 1, 1);
    cfg.dynamicSmemBytes = CfgPair::SMEM_BYTES;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<CfgPair>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// L2 hints of the operand loads (GemmParams::keep_a): by default both
// operands evict-last, since every panel is re-read by the other tiles of
// its wave (measured at 8192^3: 845 MB of DRAM reads per launch, against
// 1224 MB when the less re-read operand was marked evict-first), except an
// operand that only one tile reads: with a single tile column every panel
// of A is read once, with a single row block every panel of B. The option
// can still mark either one evict-first.
int32_t keep_a_operand(const mpgemm_plan_t& plan, int32_t l2_keep) {
    if (l2_keep == 1) return 1;
    if (l2_keep == 2) return 0;
    if (plan.n_tiles == 1 && plan.m_tiles > 1) return 0;
    if (plan.m_tiles == 1 && plan.n_tiles > 1) return 1;
    return 2;
}

// All kernel attributes the launches need, for the current device.
cudaError_t prepare_kernels() {
    cudaError_t e = set_smem_attr<Cfg256>();
    if (e == cudaSuccess) e = set_smem_attr<Cfg128>();
    if (e == cudaSuccess) e = set_smem_attr<Cfg320>();
    if (e == cudaSuccess) e = set_smem_attr<CfgPair>();
    if (e == cudaSuccess) e = set_smem_attr<CfgWide>();
    if (e == cudaSuccess) e = set_smem_attr<Cfg256K>();
    if (e == cudaSuccess) e = set_smem_attr<Cfg128K>();
    if (e == cudaSuccess) e = set_smem_attr<Cfg320K>();
    if (e == cudaSuccess) e = set_smem_attr<CfgPairK>();
    if (e == cudaSuccess) e = set_smem_attr<CfgWideK>();
    if (e == cudaSuccess) e = set_smem_attr<CfgPair384>();
    if (e == cudaSuccess) e = set_smem_attr<CfgPair384K>();
    if (e == cudaSuccess) e = set_smem_attr<CfgPair320>();
    if (e == cudaSuccess) e = set_smem_attr<CfgPair288>();
    if (e == cudaSuccess) e = set_smem_attr<CfgPair288A>();
    if (e == cudaSuccess) e = set_smem_attr<Cfg128C>();
    if (e == cudaSuccess) e = set_smem_attr<Cfg128KC>();
    return e;
}

// The A tensor maps (one per row class) and the class fields of the kernel
// parameters, for A as the kernel will read it (staged or not).
bool encode_a(const mpgemm_plan_t& plan, const void* a_use, int64_t lda_use, int64_t M, int64_t K,
              TensorMaps* maps, GemmParams* gp, MapCache* cache = nullptr) {
    const AClassLayout L = a_class_layout(a_use, lda_use, M, plan.a_classes, plan.tile_m);
    // the classes' geometry in closed form (see GemmParams)
    gp->a_classes = L.P;
    gp->a_unit = L.unit;
    gp->a_off0 = static_cast<int32_t>(reinterpret_cast<uintptr_t>(a_use) % static_cast<uintptr_t>(L.unit));
    gp->a_step = static_cast<int32_t>((2 * lda_use) % L.unit);
    gp->a_rem = static_cast<int32_t>(M % L.P);
    gp->a_rows_lo = static_cast<int32_t>(M / L.P);
    gp->a_rows_hi = gp->a_rows_lo + 1;
    gp->a_tiles_lo = static_cast<int32_t>(ceil_div(gp->a_rows_lo, plan.tile_m));
    gp->a_tiles_hi = static_cast<int32_t>(ceil_div(gp->a_rows_hi, plan.tile_m));
    if (plan.a_classes == 0) gp->a_off0 = gp->a_step = 0;   // read in place: no shift
    // (and as tables, for the kernels with room for 8 classes)
    for (int32_t r = 0; r < kTableAClasses; ++r) {
        gp->a_shift[r] = r < L.P ? L.shift[r] : 0;
        gp->a_class_rows[r] = r < L.P ? static_cast<int32_t>(L.rows[r]) : 0;
        gp->a_class_first_tile[r] = static_cast<int32_t>(L.first_tile[std::min(r, L.P)]);
    }
    gp->a_class_first_tile[kTableAClasses] = static_cast<int32_t>(L.first_tile[std::min(kTableAClasses, L.P)]);
    // (every map a kernel receives is defined: the first 8, or all when
    // there are more classes; C's and B's narrow maps are set later if used)
    std::memset(maps->a, 0, sizeof(maps->a[0]) * static_cast<size_t>(L.P > 8 ? kMaxAClasses : 8));
    std::memset(&maps->c, 0, sizeof(maps->c));
    std::memset(&maps->b_tail, 0, sizeof(maps->b_tail));
    // more classes than the per-map entries hold: the whole set at once
    const bool as_set = cache && L.P > MapCache::kEntries / 2;
    const uint64_t set_key[6] = {static_cast<uint64_t>(L.P), reinterpret_cast<uintptr_t>(a_use),
                                 static_cast<uint64_t>(lda_use), static_cast<uint64_t>(M),
                                 static_cast<uint64_t>(K), 0};
    if (as_set && cache->find_set(set_key, maps->a)) return true;
    for (int32_t r = 0; r < L.P; ++r) {
        if (L.rows[r] == 0) continue;
        if (!encode_f16(&maps->a[r], reinterpret_cast<const void*>(L.base[r]), L.rows[r], K + L.shift[r],
                        L.P * lda_use, 64, 128, as_set ? nullptr : cache))
            return false;
    }
    if (as_set) cache->put_set(set_key, maps->a, L.P);
    return true;
}

// Row-major FP32 matrix rows x cols with pitch ld (elements), 32 x 32 boxes,
// 128-byte swizzle: the tiled TMA store of the epilogue's chunks.
bool encode_f32_store(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                      MapCache* cache = nullptr, uint32_t box_cols = 32) {
    // (32 x 16 boxes, for 16-column chunks: the 64-byte swizzle)
    const CUtensorMapSwizzle swizzle = box_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const uint64_t key[6] = {32, reinterpret_cast<uintptr_t>(base), static_cast<uint64_t>(rows),
                             static_cast<uint64_t>(cols), static_cast<uint64_t>(ld),
                             (static_cast<uint64_t>(box_cols) << 32) | 32u};
    if (cache && cache->find(key, map)) return true;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    const cuuint32_t box[2] = {box_cols, 32};
    const cuuint32_t estr[2] = {1, 1};
    const bool ok = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    if (ok && cache) cache->put(key, *map);
    return ok;
}

// Let the epilogue write C with TMA when it can: C is only written
// (beta == 0), or split-K slices add into it (TMA reduce-add: C already
// holds beta * C), its rows are contiguous (one row class), its base and
// pitch are 16-byte aligned, and N is a multiple of 4. A TMA store clips a
// row only at 16-byte granularity: measured on GB300, with N = 1025 the
// store of the chunk at column 1024 also wrote columns 1025-1027 of every
// row (the padding of C). Otherwise, or when c_store forbids it, every lane
// stores (or atomically adds) its own column.
void encode_c(const mpgemm_plan_t& plan, float* C, int64_t M, int64_t N, int64_t ldc, float beta,
              int32_t c_store, TensorMaps* maps, GemmParams* gp, MapCache* cache = nullptr) {
    gp->c_tma = 0;
    if (c_store == 1 || (beta != 0.0f && plan.k_splits <= 1) || gp->a_classes != 1 || N % 4 != 0) return;
    if (plan.split_reduce) return;   // the cluster's sums are written per lane
    if (!aligned16(C, ldc, 4)) return;
    // (the 256 x 288 pair's 16-column chunks, with A read as it is: boxes of 16 columns)
    const uint32_t box_cols = (plan.tile_m == 256 && plan.tile_n == 288 && plan.tile_k == 128) ? 16 : 32;
    if (encode_f32_store(&maps->c, C, M, N, ldc, cache, box_cols)) gp->c_tma = 1;
}

// The narrow B boxes of 256 x 320 and 256 x 288 pair tiles (32 or 16 columns
// of 64 K-rows, 64- or 32-byte swizzle: the last 64- or 32-column part, half
// per CTA); nothing for other tiles.
bool encode_b_tail(const mpgemm_plan_t& plan, const void* b_use, int64_t K, int64_t N, int64_t ldb_use,
                   TensorMaps* maps, MapCache* cache = nullptr) {
    if (plan.tile_m != 256 || (plan.tile_n != 320 && plan.tile_n != 288)) return true;
    if (plan.tile_n == 288)
        return encode_f16(&maps->b_tail, b_use, K, N, ldb_use, 16, 64, cache, CU_TENSOR_MAP_SWIZZLE_32B);
    return encode_f16(&maps->b_tail, b_use, K, N, ldb_use, 32, 64, cache, CU_TENSOR_MAP_SWIZZLE_64B);
}

GemmParams make_params(const mpgemm_plan_t& plan, int64_t M, int64_t N, int64_t K, float alpha,
                       float beta, float* C, int64_t ldc, int32_t* status, uint64_t wait_limit_ns,
                       int32_t test_stall, int32_t keep_a) {
    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.M = static_cast<int32_t>(M);
    gp.N = static_cast<int32_t>(N);
    gp.K = static_cast<int32_t>(K);
    gp.m_tiles = plan.m_tiles;
    gp.n_tiles = plan.n_tiles;
    gp.k_blocks = plan.k_blocks;
    gp.tiles = static_cast<int32_t>(plan.tiles);
    gp.tail_start = static_cast<int32_t>(plan.tiles - plan.split_tiles);
    gp.items = static_cast<int32_t>(plan.items);
    gp.k_splits = plan.k_splits;
    gp.kb_per_split = static_cast<int32_t>(ceil_div(plan.k_blocks, plan.k_splits));
    gp.raster_group = plan.raster_group;
    gp.alpha = alpha;
    gp.beta = beta;
    gp.C = C;
    gp.ldc = ldc;
    gp.status = status;
    gp.wait_limit_ns = wait_limit_ns;
    gp.test_stall = test_stall;
    gp.keep_a = keep_a;
    // split-K slices after the pass that applies beta (launch_plan)
    gp.overlap_prepass = (plan.k_splits > 1 && !plan.split_reduce && beta != 1.0f) ? 1 : 0;
    if (plan.sk_ranges > 0) {   // (the caller sets sk_flags and sk_epoch)
        gp.sk_units = static_cast<int32_t>(plan.tiles * plan.k_blocks);
        gp.sk_ranges = plan.sk_ranges;
        const std::vector<int32_t> start = sk_range_starts(gp.sk_units, plan.k_blocks, plan.sk_ranges);
        std::copy(start.begin(), start.end(), gp.sk_start);
    }
    return gp;
}

cudaError_t launch_plan(const mpgemm_plan_t& plan, bool b_col_major, int max_clusters,
                        const TensorMaps& ta, const CUtensorMap& tb, const GemmParams& gp,
                        cudaStream_t stream) {
    if (plan.k_splits > 1 && !plan.split_reduce && gp.beta != 1.0f) {
        // the slices add into C: apply beta (or clear C) once, first
        scale_c<<<grid_for(static_cast<int64_t>(gp.M) * gp.N, plan.grid), 256, 0, stream>>>(
            gp.C, gp.ldc, gp.M, gp.N, gp.beta);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (plan.tile_m == 256) {
        int grid = plan.grid;
        if (max_clusters > 0 && grid > 2 * max_clusters) grid = 2 * max_clusters;
        // every stream-K range needs its own pair, all resident together
        if (plan.sk_ranges > 0 && (grid != 2 * plan.sk_ranges || !gp.sk_flags || gp.sk_epoch == 0))
            return cudaErrorInvalidValue;
        if (plan.tile_n == 512)
            return b_col_major ? launch_tc<CfgWideK>(grid, ta, tb, gp, stream)
                               : launch_tc<CfgWide>(grid, ta, tb, gp, stream);
        if (plan.tile_n == 384)
            return b_col_major ? launch_tc<CfgPair384K>(grid, ta, tb, gp, stream)
                               : launch_tc<CfgPair384>(grid, ta, tb, gp, stream);
        if (plan.tile_n == 320) return launch_tc<CfgPair320>(grid, ta, tb, gp, stream);
        if (plan.tile_n == 288)
            return plan.tile_k == 128 ? launch_tc<CfgPair288A>(grid, ta, tb, gp, stream)
                                      : launch_tc<CfgPair288>(grid, ta, tb, gp, stream);
        return b_col_major ? launch_tc<CfgPairK>(grid, ta, tb, gp, stream)
                           : launch_tc<CfgPair>(grid, ta, tb, gp, stream);
    }
    if (plan.split_reduce) {
        // one cluster of k_splits CTAs per tile, every CTA one slice
        if (plan.tile_n != 128 || plan.k_splits < 2 || plan.k_splits > kMaxClusterSplits ||
            static_cast<int64_t>(plan.grid) != plan.items)
            return cudaErrorInvalidValue;
        return b_col_major ? launch_tc<Cfg128KC>(plan.grid, ta, tb, gp, stream)
                           : launch_tc<Cfg128C>(plan.grid, ta, tb, gp, stream);
    }
    if (plan.tile_n == 320)
        return b_col_major ? launch_tc<Cfg320K>(plan.grid, ta, tb, gp, stream)
                           : launch_tc<Cfg320>(plan.grid, ta, tb, gp, stream);
    if (plan.tile_n == 256)
        return b_col_major ? launch_tc<Cfg256K>(plan.grid, ta, tb, gp, stream)
                           : launch_tc<Cfg256>(plan.grid, ta, tb, gp, stream);
    return b_col_major ? launch_tc<Cfg128K>(plan.grid, ta, tb, gp, stream)
                       : launch_tc<Cfg128>(plan.grid, ta, tb, gp, stream);
}

}  // namespace
}  // namespace mpgemm

using namespace mpgemm;

struct mpgemm_handle_st;

namespace {
// mpgemm_solve's handle per device, created by the first call on that device
// that succeeds in creating it (a failed creation is returned and the next
// call tries again) and kept until the process exits.
constexpr int kSolveMaxDevices = 64;
struct SolveDevice {
    mpgemm_handle_st* handle = nullptr;
    std::mutex mu;   // guards `handle`; its host state (tensor-map cache, workspace) is not thread-safe
};
SolveDevice g_solve_devices[kSolveMaxDevices];
}  // namespace

struct mpgemm_handle_st {
    MapCache map_cache;              // tensor maps of recent calls
    int device = 0;
    int num_sms = 0;
    int max_clusters = 0;            // CTA pairs of the pair kernel resident at once
    Options opt;
    int32_t* status_host = nullptr;  // mapped pinned memory: {code, role, block, detail}
    int32_t* status_dev = nullptr;
    void* ws = nullptr;              // staging copies of unaligned operands
    size_t ws_bytes = 0;
    void* host_ws = nullptr;         // device copies for mpgemm_run_host
    size_t host_ws_bytes = 0;
    int32_t* sk_flags = nullptr;     // stream-K flags (zeroed when allocated), and the epoch of
    size_t sk_flags_bytes = 0;       // the last call that used them
    int32_t sk_epoch = 0;
};

namespace {

mpgemm_status_t ensure_buffer(void** ptr, size_t* cap, size_t need, cudaStream_t s) {
    if (need <= *cap) return MPGEMM_OK;
    if (*ptr) cudaFreeAsync(*ptr, s);
    *ptr = nullptr;
    *cap = 0;
    if (cudaMallocAsync(ptr, need, s) != cudaSuccess) {
        cudaGetLastError();
        *ptr = nullptr;
        return MPGEMM_ERR_ALLOC;
    }
    *cap = need;
    return MPGEMM_OK;
}

// The tensor-map encoder is a driver-API call and needs the device's
// context current in the calling thread. The runtime binds a thread to the
// device's primary context lazily, at its first call that needs one, so a
// thread whose first GEMM needs no other runtime call before the encoder
// (no staging copy, no workspace to grow) would meet it unbound. Bind it
// here, once per thread and device; `dev` is already the current device,
// so the caller's choice of device is not changed.
bool bind_context(int dev) {
    thread_local int bound = -1;
    if (bound == dev) return true;
    if (cudaSetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    bound = dev;
    return true;
}

// The handle's device must be current (it owns the workspace and the launch
// configuration of that device).
mpgemm_status_t enter_device(const mpgemm_handle_st* h) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    if (cur != h->device) return MPGEMM_ERR_INVALID_VALUE;
    return bind_context(cur) ? MPGEMM_OK : MPGEMM_ERR_CUDA;
}

mpgemm_status_t take_device_report(mpgemm_handle_t h, int32_t info[4]) {
    volatile int32_t* s = h->status_host;
    const int32_t code = s[0];
    if (info) {
        info[0] = code;
        info[1] = code ? s[1] : 0;
        info[2] = code ? s[2] : 0;
        info[3] = code ? s[3] : 0;
    }
    if (code == 0) return MPGEMM_OK;
    s[1] = s[2] = s[3] = 0;
    s[0] = 0;
    return MPGEMM_ERR_DEVICE_TIMEOUT;
}

}  // namespace

extern "C" {

const char* mpgemm_status_string(mpgemm_status_t s) {
    switch (s) {
        case MPGEMM_OK: return "success";
        case MPGEMM_ERR_INVALID_VALUE: return "invalid argument";
        case MPGEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
        case MPGEMM_ERR_ALLOC: return "allocation failed";
        case MPGEMM_ERR_LAUNCH: return "kernel launch or copy failed";
        case MPGEMM_ERR_DEVICE_TIMEOUT: return "a bounded device wait gave up";
        case MPGEMM_ERR_CUDA: return "CUDA error";
        case MPGEMM_ERR_SCRATCH_LIMIT:
            return "operands need more staging scratch than mpgemm_run_noalloc's fixed area holds";
    }
    return "unknown status";
}

mpgemm_status_t mpgemm_plan(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                            int64_t lda, const void* B, int64_t ldb, float beta, const float* C,
                            int64_t ldc, int32_t num_sms, int32_t tile_m, int32_t tile_n,
                            int32_t max_ctas, int32_t force_staging, int32_t b_col_major,
                            mpgemm_plan_t* out) {
    if (!out) return MPGEMM_ERR_INVALID_VALUE;
    if (tile_m != 0 && tile_m != 128 && tile_m != 256) return MPGEMM_ERR_INVALID_VALUE;
    if (tile_n != 0 && tile_n != 128 && tile_n != 256 && tile_n != 288 && tile_n != 320 && tile_n != 384 &&
        tile_n != 512)
        return MPGEMM_ERR_INVALID_VALUE;
    if (max_ctas < 0) return MPGEMM_ERR_INVALID_VALUE;
    Options opt;
    opt.tile_m = tile_m;
    opt.tile_n = tile_n;
    opt.max_ctas = max_ctas;
    opt.b_col_major = b_col_major ? 1 : 0;
    opt.force_staging = force_staging ? 1 : 0;
    return make_plan(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, num_sms, opt, out);
}

mpgemm_status_t mpgemm_create(mpgemm_handle_t* out) {
    if (!out) return MPGEMM_ERR_INVALID_VALUE;
    *out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MPGEMM_ERR_UNSUPPORTED_DEVICE;
    if (!encode_fn()) return MPGEMM_ERR_CUDA;
    if (prepare_kernels() != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    mpgemm_handle_st* h = new (std::nothrow) mpgemm_handle_st();
    if (!h) return MPGEMM_ERR_ALLOC;
    h->device = dev;
    h->num_sms = sms;
    h->max_clusters = max_pair_clusters();
    void* st = nullptr;
    if (cudaHostAlloc(&st, 4 * sizeof(int32_t), cudaHostAllocMapped) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return MPGEMM_ERR_ALLOC;
    }
    h->status_host = static_cast<int32_t*>(st);
    std::memset(h->status_host, 0, 4 * sizeof(int32_t));
    void* dptr = nullptr;
    if (cudaHostGetDevicePointer(&dptr, st, 0) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeHost(st);
        delete h;
        return MPGEMM_ERR_CUDA;
    }
    h->status_dev = static_cast<int32_t*>(dptr);
    *out = h;
    return MPGEMM_OK;
}

mpgemm_status_t mpgemm_destroy(mpgemm_handle_t h) {
    if (!h) return MPGEMM_OK;
    if (h->ws) cudaFree(h->ws);
    if (h->host_ws) cudaFree(h->host_ws);
    if (h->sk_flags) cudaFree(h->sk_flags);
    if (h->status_host) cudaFreeHost(h->status_host);
    cudaGetLastError();
    delete h;
    return MPGEMM_OK;
}

mpgemm_status_t mpgemm_set_option(mpgemm_handle_t h, mpgemm_option_t opt, int64_t value) {
    if (!h) return MPGEMM_ERR_INVALID_VALUE;
    switch (opt) {
        case MPGEMM_OPT_TILE_N:
            if (value != 0 && value != 128 && value != 256 && value != 288 && value != 320 && value != 384 &&
                value != 512)
                return MPGEMM_ERR_INVALID_VALUE;
            h->opt.tile_n = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_MAX_CTAS:
            if (value < 0 || value > kDimLimit) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.max_ctas = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_FORCE_STAGING:
            if (value != 0 && value != 1) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.force_staging = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_WAIT_LIMIT_US:
            if (value < 1000 || value > 60000000) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.wait_limit_ns = static_cast<uint64_t>(value) * 1000ull;
            return MPGEMM_OK;
        case MPGEMM_OPT_RASTER_GROUP:
            if (value < 0 || value > 65536) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.raster_group = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_L2_KEEP:
            if (value < 0 || value > 2) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.l2_keep = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_SPLIT_K:
            if (value < 0 || value > 64) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.split_k = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_TILE_M:
            if (value != 0 && value != 128 && value != 256) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.tile_m = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_TEST_STALL:
            if (value != 0 && value != 1) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.test_stall = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_C_STORE:
            if (value != 0 && value != 1) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.c_store = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_ACCUMULATOR:
            if (value != 0 && value != 16 && value != 32) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.acc16 = value == 16 ? 1 : 0;
            return MPGEMM_OK;
        case MPGEMM_OPT_REPRODUCIBLE:
            if (value != 0 && value != 1) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.reproducible = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_STREAM_K:
            if (value < 0 || value > 2) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.stream_k = static_cast<int32_t>(value);
            return MPGEMM_OK;
        case MPGEMM_OPT_SPLIT_REDUCE:
            if (value < 0 || value > 2) return MPGEMM_ERR_INVALID_VALUE;
            h->opt.split_reduce = static_cast<int32_t>(value);
            return MPGEMM_OK;
    }
    return MPGEMM_ERR_INVALID_VALUE;
}

mpgemm_status_t mpgemm_plan_call(mpgemm_handle_t h, mpgemm_b_layout_t b_layout, int64_t M, int64_t N,
                                 int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                                 int64_t ldb, float beta, const float* C, int64_t ldc, mpgemm_plan_t* out) {
    if (!h || !out) return MPGEMM_ERR_INVALID_VALUE;
    if (b_layout != MPGEMM_B_ROW_MAJOR && b_layout != MPGEMM_B_COL_MAJOR) return MPGEMM_ERR_INVALID_VALUE;
    if (mpgemm_status_t st0 = enter_device(h); st0 != MPGEMM_OK) return st0;
    Options opt = h->opt;
    opt.pair_units = h->max_clusters;
    opt.b_col_major = b_layout == MPGEMM_B_COL_MAJOR ? 1 : 0;
    return make_plan(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, h->num_sms, opt, out);
}

mpgemm_status_t mpgemm_run_ex(mpgemm_handle_t h, mpgemm_b_layout_t b_layout, int64_t M, int64_t N,
                              int64_t K, float alpha, const void* A, int64_t lda, const void* B,
                              int64_t ldb, float beta, float* C, int64_t ldc, void* stream_ptr) {
    if (!h) return MPGEMM_ERR_INVALID_VALUE;
    if (b_layout != MPGEMM_B_ROW_MAJOR && b_layout != MPGEMM_B_COL_MAJOR) return MPGEMM_ERR_INVALID_VALUE;
    const bool b_col = (b_layout == MPGEMM_B_COL_MAJOR);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    mpgemm_plan_t plan;
    Options opt = h->opt;
    if (mpgemm_status_t st0 = enter_device(h); st0 != MPGEMM_OK) return st0;
    opt.pair_units = h->max_clusters;
    opt.b_col_major = b_col ? 1 : 0;
    mpgemm_status_t st = make_plan(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, h->num_sms, opt, &plan);
    if (st != MPGEMM_OK) return st;
    if (take_device_report(h, nullptr) != MPGEMM_OK) return MPGEMM_ERR_DEVICE_TIMEOUT;
    if (plan.quick == 1) return MPGEMM_OK;
    if (plan.quick == 2) {
        scale_c<<<grid_for(M * N, h->num_sms), 256, 0, stream>>>(C, ldc, M, N, beta);
        return cudaGetLastError() == cudaSuccess ? MPGEMM_OK : MPGEMM_ERR_LAUNCH;
    }

    const void* a_use = A;
    const void* b_use = B;
    int64_t lda_use = lda, ldb_use = ldb;
    if (plan.workspace_bytes > 0) {
        st = ensure_buffer(&h->ws, &h->ws_bytes, static_cast<size_t>(plan.workspace_bytes), stream);
        if (st != MPGEMM_OK) return st;
        uint8_t* ws = static_cast<uint8_t*>(h->ws);
        if (plan.stage_a) {
            lda_use = round_up(K, 8);
            stage_rows_u16<<<grid_for(M * ceil_div(K, 8), h->num_sms), 256, 0, stream>>>(
                static_cast<const uint16_t*>(A), lda, reinterpret_cast<uint16_t*>(ws), lda_use, M, K);
            a_use = ws;
            ws += round_up(M * lda_use * 2, 256);
        }
        if (plan.stage_b) {
            // B as stored: K rows of N (row-major) or N rows of K (column-major)
            const int64_t b_rows = b_col ? N : K, b_cols = b_col ? K : N;
            ldb_use = round_up(b_cols, 8);
            stage_rows_u16<<<grid_for(b_rows * ceil_div(b_cols, 8), h->num_sms), 256, 0, stream>>>(
                static_cast<const uint16_t*>(B), ldb, reinterpret_cast<uint16_t*>(ws), ldb_use, b_rows,
                b_cols);
            b_use = ws;
        }
        if (cudaGetLastError() != cudaSuccess) return MPGEMM_ERR_LAUNCH;
    }

    CUtensorMap tb;
    if (!(b_col ? encode_f16(&tb, b_use, N, K, ldb_use, 64, 64, &h->map_cache)
                : encode_f16(&tb, b_use, K, N, ldb_use, 64, 64, &h->map_cache)))
        return MPGEMM_ERR_CUDA;

    GemmParams gp = make_params(plan, M, N, K, alpha, beta, C, ldc, h->status_dev,
                                h->opt.wait_limit_ns, h->opt.test_stall,
                                keep_a_operand(plan, h->opt.l2_keep));
    TensorMaps ta;
    if (!encode_a(plan, a_use, lda_use, M, K, &ta, &gp, &h->map_cache)) return MPGEMM_ERR_CUDA;
    if (!encode_b_tail(plan, b_use, K, N, ldb_use, &ta, &h->map_cache)) return MPGEMM_ERR_CUDA;
    encode_c(plan, C, M, N, ldc, beta, h->opt.c_store, &ta, &gp, &h->map_cache);
    gp.acc16 = h->opt.acc16;
    if (plan.sk_ranges > 0) {
        // Stream-K flags: one per range, CTA and epilogue warp. A new buffer
        // starts at zero, which no call's epoch is; each call publishes a
        // new epoch, so flags left by earlier calls never match.
        const size_t need = static_cast<size_t>(plan.sk_ranges) * kSkFlagsPerRange * sizeof(int32_t);
        if (need > h->sk_flags_bytes || h->sk_epoch == INT32_MAX) {
            void* buf = h->sk_flags;
            size_t cap = h->sk_flags_bytes;
            st = ensure_buffer(&buf, &cap, need, stream);
            h->sk_flags = static_cast<int32_t*>(buf);
            h->sk_flags_bytes = cap;
            if (st != MPGEMM_OK) return st;
            if (cudaMemsetAsync(h->sk_flags, 0, h->sk_flags_bytes, stream) != cudaSuccess) {
                cudaGetLastError();
                return MPGEMM_ERR_LAUNCH;
            }
            h->sk_epoch = 0;
        }
        gp.sk_flags = h->sk_flags;
        gp.sk_epoch = ++h->sk_epoch;
    }
    if (launch_plan(plan, b_col, h->max_clusters, ta, tb, gp, stream) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_LAUNCH;
    }
    return MPGEMM_OK;
}

mpgemm_status_t mpgemm_run(mpgemm_handle_t h, int64_t M, int64_t N, int64_t K, float alpha,
                           const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                           float* C, int64_t ldc, void* stream_ptr) {
    return mpgemm_run_ex(h, MPGEMM_B_ROW_MAJOR, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                         stream_ptr);
}

mpgemm_status_t mpgemm_run_host(mpgemm_handle_t h, int64_t M, int64_t N, int64_t K, float alpha,
                                const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                                float* C, int64_t ldc, void* stream_ptr) {
    if (!h) return MPGEMM_ERR_INVALID_VALUE;
    mpgemm_status_t st = validate(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (st != MPGEMM_OK) return st;
    if (M == 0 || N == 0) return MPGEMM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const bool need_ab = (K > 0 && alpha != 0.0f);
    // Every operand travels verbatim with its own pitch, as one contiguous
    // copy (one large DMA instead of one per row); mpgemm_run then stages A
    // or B on the device if that pitch breaks the 16-byte rule, and the
    // epilogue writes C at any pitch. Only when beta == 0 and C has padding
    // columns is C copied back row by row, so the host's padding columns
    // (never sent to the device) are not overwritten.
    const int64_t a_elems = need_ab ? (M - 1) * lda + K : 0;
    const int64_t b_elems = need_ab ? (K - 1) * ldb + N : 0;
    const int64_t c_elems = (M - 1) * ldc + N;
    const int64_t ldc_d = ldc;
    const int64_t a_bytes = round_up(a_elems * 2, 256);
    const int64_t b_bytes = round_up(b_elems * 2, 256);
    const int64_t c_bytes = round_up(c_elems * 4, 256);
    st = ensure_buffer(&h->host_ws, &h->host_ws_bytes, static_cast<size_t>(a_bytes + b_bytes + c_bytes),
                       stream);
    if (st != MPGEMM_OK) return st;
    uint8_t* base = static_cast<uint8_t*>(h->host_ws);
    void* dA = base;
    void* dB = base + a_bytes;
    float* dC = reinterpret_cast<float*>(base + a_bytes + b_bytes);
    if (need_ab) {
        if (cudaMemcpyAsync(dA, A, static_cast<size_t>(a_elems) * 2, cudaMemcpyHostToDevice, stream) !=
                cudaSuccess ||
            cudaMemcpyAsync(dB, B, static_cast<size_t>(b_elems) * 2, cudaMemcpyHostToDevice, stream) !=
                cudaSuccess) {
            cudaGetLastError();
            return MPGEMM_ERR_LAUNCH;
        }
    }
    if (beta != 0.0f &&
        cudaMemcpyAsync(dC, C, static_cast<size_t>(c_elems) * 4, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_LAUNCH;
    }
    st = mpgemm_run(h, M, N, K, alpha, need_ab ? dA : nullptr, need_ab ? lda : (K > 1 ? K : 1),
                    need_ab ? dB : nullptr, need_ab ? ldb : (N > 1 ? N : 1), beta, dC, ldc_d, stream_ptr);
    if (st != MPGEMM_OK) return st;
    const cudaError_t back =
        (beta != 0.0f || ldc == N)
            ? cudaMemcpyAsync(C, dC, static_cast<size_t>(c_elems) * 4, cudaMemcpyDeviceToHost, stream)
            : cudaMemcpy2DAsync(C, ldc * 4, dC, ldc_d * 4, N * 4, M, cudaMemcpyDeviceToHost, stream);
    if (back != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_LAUNCH;
    }
    return MPGEMM_OK;
}

mpgemm_status_t mpgemm_solve(const void* a, const void* b, float* c, size_t m, size_t n, size_t k,
                             void* stream) {
    if (m > static_cast<size_t>(kDimLimit) || n > static_cast<size_t>(kDimLimit) ||
        k > static_cast<size_t>(kDimLimit))
        return MPGEMM_ERR_INVALID_VALUE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kSolveMaxDevices) return MPGEMM_ERR_CUDA;
    SolveDevice& d = g_solve_devices[dev];
    const int64_t M = static_cast<int64_t>(m), N = static_cast<int64_t>(n), K = static_cast<int64_t>(k);
    std::lock_guard<std::mutex> lock(d.mu);
    if (!d.handle) {
        mpgemm_handle_st* h = nullptr;
        const mpgemm_status_t st = mpgemm_create(&h);
        if (st != MPGEMM_OK) return st;
        d.handle = h;
    }
    return mpgemm_run_ex(d.handle, MPGEMM_B_COL_MAJOR, M, N, K, 1.0f, a, K > 1 ? K : 1, b,
                         K > 1 ? K : 1, 0.0f, c, N > 1 ? N : 1, stream);
}

mpgemm_status_t mpgemm_probe_mma_rate(int32_t ctas, int32_t mmas, uint64_t* out, void* stream) {
    if (ctas < 1 || ctas > 65535 || mmas < 4 || mmas > (1 << 22) || !out ||
        reinterpret_cast<uintptr_t>(out) % 8 != 0)
        return MPGEMM_ERR_INVALID_VALUE;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MPGEMM_ERR_UNSUPPORTED_DEVICE;
    if (cudaFuncSetAttribute(mma_rate_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmemBytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    mma_rate_probe<<<ctas, 32, kProbeSmemBytes, static_cast<cudaStream_t>(stream)>>>(
        mmas, kDefaultWaitLimitNs, reinterpret_cast<unsigned long long*>(out));
    if (cudaGetLastError() != cudaSuccess) return MPGEMM_ERR_LAUNCH;
    return MPGEMM_OK;
}

mpgemm_status_t mpgemm_sync_status(mpgemm_handle_t h, void* stream, int32_t info[4]) {
    if (!h) return MPGEMM_ERR_INVALID_VALUE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    return take_device_report(h, info);
}

}  // extern "C"

// ------------------------------------------------------------------ no-allocation entry point
//
// mpgemm_run_noalloc serves callers that cannot allocate (see the header):
// the staging copies that mpgemm_run puts in a handle's workspace go into a
// fixed file-scope device array instead, and the bounded-wait status words
// live at its start. In host code `g_noalloc_scratch` is only a host-side
// stand-in for the symbol: the kernels get the device address that
// cudaGetSymbolAddress returns for the current device, looked up once per
// device on that device's first call.

namespace {

constexpr int64_t kNoAllocScratchBytes = MPGEMM_NOALLOC_SCRATCH_BYTES;
constexpr int64_t kNoAllocStatusBytes = 256;  // 4 status words, padded to keep staging aligned
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocStatusBytes + kNoAllocScratchBytes];

struct NoAllocDevice {
    std::mutex mu;
    bool ready = false;                // set once a set-up has succeeded
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int max_clusters = 0;
};

NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];

// With that device current: look up the scratch array's device address and
// set the kernels' attributes. Called until it succeeds once per device (a
// failure, e.g. an error another component left pending, is returned and
// the next call tries again).
mpgemm_status_t noalloc_setup(NoAllocDevice& d, int dev) {
    std::lock_guard<std::mutex> lock(d.mu);
    if (d.ready) return MPGEMM_OK;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MPGEMM_ERR_UNSUPPORTED_DEVICE;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr ||
        !encode_fn() || prepare_kernels() != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_CUDA;
    }
    d.scratch = static_cast<unsigned char*>(ptr);
    d.num_sms = sms;
    d.max_clusters = max_pair_clusters();
    d.ready = true;
    return MPGEMM_OK;
}

}  // namespace

extern "C" mpgemm_status_t mpgemm_run_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                              const void* A, int64_t lda, const void* B,
                                              int64_t ldb, float beta, float* C, int64_t ldc,
                                              void* stream_ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (dev < 0 || dev >= kNoAllocMaxDevices) return MPGEMM_ERR_CUDA;
    NoAllocDevice& d = g_noalloc_devices[dev];
    if (mpgemm_status_t s0 = noalloc_setup(d, dev); s0 != MPGEMM_OK) return s0;
    if (!bind_context(dev)) return MPGEMM_ERR_CUDA;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    Options opt;  // defaults: automatic tile width, one CTA per SM, 4 s wait limit
    opt.pair_units = d.max_clusters;
    opt.stream_k = 1;   // (its flags would need memory of their own)
    mpgemm_plan_t plan;
    mpgemm_status_t st =
        make_plan(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, d.num_sms, opt, &plan);
    if (st != MPGEMM_OK) return st;
    if (plan.quick == 1) return MPGEMM_OK;
    if (plan.quick == 2) {
        scale_c<<<grid_for(M * N, d.num_sms), 256, 0, stream>>>(C, ldc, M, N, beta);
        return cudaGetLastError() == cudaSuccess ? MPGEMM_OK : MPGEMM_ERR_LAUNCH;
    }
    if (plan.workspace_bytes > kNoAllocScratchBytes) return MPGEMM_ERR_SCRATCH_LIMIT;

    // The status words must start at zero; the array keeps the last call's contents.
    int32_t* status = reinterpret_cast<int32_t*>(d.scratch);
    if (cudaMemsetAsync(status, 0, 4 * sizeof(int32_t), stream) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_LAUNCH;
    }
    // (B is row-major here, so an unaligned A is read in row classes and
    // never staged: only B's copy uses the scratch)
    if (plan.stage_a) return MPGEMM_ERR_INVALID_VALUE;
    const void* a_use = A;
    const void* b_use = B;
    const int64_t lda_use = lda;
    int64_t ldb_use = ldb;
    unsigned char* ws = d.scratch + kNoAllocStatusBytes;
    if (plan.stage_b) {
        ldb_use = round_up(N, 8);
        stage_rows_u16<<<grid_for(K * ceil_div(N, 8), d.num_sms), 256, 0, stream>>>(
            static_cast<const uint16_t*>(B), ldb, reinterpret_cast<uint16_t*>(ws), ldb_use, K, N);
        b_use = ws;
    }
    if (cudaGetLastError() != cudaSuccess) return MPGEMM_ERR_LAUNCH;

    CUtensorMap tb;
    if (!encode_f16(&tb, b_use, K, N, ldb_use, 64, 64)) return MPGEMM_ERR_CUDA;
    GemmParams gp = make_params(plan, M, N, K, alpha, beta, C, ldc, status, opt.wait_limit_ns, 0,
                                keep_a_operand(plan, 0));
    TensorMaps ta;
    if (!encode_a(plan, a_use, lda_use, M, K, &ta, &gp)) return MPGEMM_ERR_CUDA;
    if (!encode_b_tail(plan, b_use, K, N, ldb_use, &ta)) return MPGEMM_ERR_CUDA;
    encode_c(plan, C, M, N, ldc, beta, 0, &ta, &gp);
    if (launch_plan(plan, false, d.max_clusters, ta, tb, gp, stream) != cudaSuccess) {
        cudaGetLastError();
        return MPGEMM_ERR_LAUNCH;
    }
    return MPGEMM_OK;
}
