// gemm_relu_kernels.cuh -- device code of the fused fp16 GEMM + ReLU.
//
//   C = fp16( max( A . B , 0 ) ),  A: M x K, B: K x N, C: M x N, row-major.
//
// The operation is the FP16 GEMM + ReLU quickstart of "TileLang 编程基本知识点"
// (section 二) and the GEMM section of "在 TileLang 中編寫高效能核心：從 GEMM 到
// MLA": fp16 tiles staged in shared memory, a K loop over BK-wide strips,
// tensor-core MMA into an fp32 accumulator, max(x, 0) on the accumulator, one
// cast to fp16 on the way out.  The pages' A100/H100 lowering (cp.async or
// TMA, mma.sync or wgmma) is replaced here by the sm_103a path the same
// page's section 四/5.4 names for datacenter Blackwell -- TMA + mbarrier
// pipeline, tcgen05.mma with a TMEM accumulator -- written by hand:
//
//   warp 0 (or warps 0-3)  producer: TMA (or predicated loads) into a ring of
//                          kStages shared-memory stages, full/empty mbarriers
//   next warp              MMA issuer: one thread issues tcgen05.mma into one
//                          of two TMEM accumulators, commits to mbarriers
//   last 4 warps           epilogue: tcgen05.ld -> ReLU -> fp16 -> swizzled
//                          shared staging -> TMA store (or predicated stores)
//
// Roles iterate the same persistent sequence of output tiles (grid = at most
// one CTA per SM, "TileLang tutorial", chapter "Persistent kernel"), taken in
// grouped order for L2 reuse (T.use_swizzle(panel_size, order="col") on the
// atlascloud page).  Every mbarrier wait is bounded by wall-clock time; on
// expiry the CTA records GEMMRELU_ERR_TIMEOUT in a device status word, every
// role leaves its loop, in-flight copies are drained and TMEM is freed.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "sm103.cuh"

namespace gemmrelu {

using namespace sm103;

// ------------------------------------------------------------------ status

// Device watchdog word: 0, or the first error code recorded since the host
// last read it.  `g_status_where` tells which wait expired (debugging aid).
__device__ unsigned int g_status;
__device__ unsigned int g_status_where;

constexpr unsigned kStatusTimeout = 5;  // == GEMMRELU_ERR_TIMEOUT

enum WaitSite : unsigned {
    kSiteProducerEmpty = 1,
    kSiteMmaAccEmpty = 2,
    kSiteMmaFull = 3,
    kSiteEpiAccFull = 4,
    kSiteDrain = 5,
    kSitePieceFlag = 6,
    kSiteClusterReduce = 7,
};

__device__ __forceinline__ void record_timeout(volatile uint32_t *abort_flag, unsigned where) {
    *abort_flag = 1u;
    if (atomicCAS(&g_status, 0u, kStatusTimeout) == 0u)
        g_status_where = where;
}

// Wait for the phase of parity `parity` of mbarrier `bar`; give up after
// `limit_ns` of wall-clock time (recording a timeout) or as soon as another
// role of this CTA has given up.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                             volatile uint32_t *abort_flag, unsigned where) {
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > limit_ns) {
            record_timeout(abort_flag, where);
            return false;
        }
    }
}

// wait_bounded with a pause of `sleep_ns` between polls: for waits that last
// a whole tile (the epilogue's), so that the waiting warps leave issue slots
// to warps that share their scheduler and do the work.
__device__ __forceinline__ bool wait_bounded_sleep(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                   volatile uint32_t *abort_flag, unsigned where,
                                                   unsigned sleep_ns) {
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > limit_ns) {
            record_timeout(abort_flag, where);
            return false;
        }
    }
}

// wait_bounded without the suspend hint (mbar_try_wait_eager): for the
// softmax <-> MMA hand-offs of the attention kernel, where the waiting
// thread's wake-up latency is on the critical path (measured: 5% there).
__device__ __forceinline__ bool wait_bounded_eager(uint32_t bar, uint32_t parity,
                                                   uint64_t limit_ns,
                                                   volatile uint32_t *abort_flag,
                                                   unsigned where) {
    if (mbar_try_wait_eager(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_eager(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > limit_ns) {
            record_timeout(abort_flag, where);
            return false;
        }
    }
}

// wait_bounded for a phase completed by other CTAs of the cluster (acquire
// at cluster scope, so their shared-memory writes before arriving are seen).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                     uint64_t limit_ns,
                                                     volatile uint32_t *abort_flag,
                                                     unsigned where) {
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > limit_ns) {
            record_timeout(abort_flag, where);
            return false;
        }
    }
}

// Same, but ignores the abort flag: used to drain work already in flight.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                           volatile uint32_t *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            record_timeout(abort_flag, kSiteDrain);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ rasteriser

// Linear tile id -> (m block, n block).  Panels of `panel` consecutive M
// blocks; inside a panel M varies fastest, then N; panels follow in M order.
// The last panel may hold fewer M blocks.  A bijection on [0, m_tiles*n_tiles).
__host__ __device__ __forceinline__ void tile_coord(int64_t t, int64_t m_tiles, int64_t n_tiles,
                                                    int64_t panel, int64_t &mb, int64_t &nb) {
    const int64_t per_panel = panel * n_tiles;
    const int64_t p = t / per_panel;
    const int64_t r = t - p * per_panel;
    const int64_t left = m_tiles - p * panel;
    const int64_t rows = left < panel ? left : panel;
    mb = p * panel + r % rows;
    nb = r / rows;
}

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint32_t relu_pack_half2(uint32_t lo_bits, uint32_t hi_bits) {
    const float lo = fmaxf(__uint_as_float(lo_bits), 0.0f);
    const float hi = fmaxf(__uint_as_float(hi_bits), 0.0f);
    const __half2 h = __floats2half2_rn(lo, hi);  // .x (low half) = lo
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_b32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Byte offset of 16-byte chunk j of row r inside a 128-byte-swizzled tile
// whose rows are 128 bytes: the chunk index is XORed with (row mod 8), the
// pattern TMA's SWIZZLE_128B mode writes and tcgen05's SWIZZLE_128B reads.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t j) {
    return r * 128u + ((j ^ (r & 7u)) << 4);
}

// ------------------------------------------------------------------ predicated loads
//
// Operands whose rows TMA cannot describe as a plain matrix (a row pitch or a
// base address that is not a multiple of 16 bytes) are staged in two steps.
// A row segment of 8 * G fp16 starts at some even byte offset `off` inside a
// 16-byte block and so spans G + 1 aligned 16-byte blocks.  First the aligned
// blocks come into a raw shared-memory slot by TMA (see RowMaps: rows r and
// r + 8 start at the same offset modulo 16, because eight rows are 16 * cols
// bytes, so each residue of the rows modulo 8 is a regular 2-D tensor with a
// 16-byte-aligned base).  Then a group of G lanes walks along each raw row:
// lane c reads blocks c and c + 1 and funnel-shifts the 32 bytes by `off` to
// get the 16 bytes of its chunk, which it stores in the operand layout.  A
// warp that takes the rows of one residue sees one offset per operand for
// the whole kernel.

// Byte offset `off` (even, 0..14) of a row segment inside its first 16-byte
// block, split for window16: word shift by 1, word shift by 2, bit shift.
struct Shift {
    bool s1, s2;
    uint32_t sh;
};

__device__ __forceinline__ Shift make_shift(uint32_t off) {
    return Shift{(off & 4u) != 0, (off & 8u) != 0, (off & 3u) * 8u};
}

// The 16 bytes at byte offset `off` of the 32 bytes v0 || v1: the word offset
// off / 4 as two selects, the half-word rest as a funnel shift.
__device__ __forceinline__ uint4 window16(const uint4 &v0, const uint4 &v1, const Shift &f) {
    const uint32_t t0 = f.s1 ? v0.y : v0.x, t1 = f.s1 ? v0.z : v0.y, t2 = f.s1 ? v0.w : v0.z;
    const uint32_t t3 = f.s1 ? v1.x : v0.w, t4 = f.s1 ? v1.y : v1.x, t5 = f.s1 ? v1.z : v1.y;
    const uint32_t t6 = f.s1 ? v1.w : v1.z;
    const uint32_t x0 = f.s2 ? t2 : t0, x1 = f.s2 ? t3 : t1, x2 = f.s2 ? t4 : t2;
    const uint32_t x3 = f.s2 ? t5 : t3, x4 = f.s2 ? t6 : t4;
    return make_uint4(__funnelshift_r(x0, x1, f.sh), __funnelshift_r(x1, x2, f.sh),
                      __funnelshift_r(x2, x3, f.sh), __funnelshift_r(x3, x4, f.sh));
}

// Predicated store of a warp's 32 rows x 64 fp16 columns of C (rows row0 ..,
// columns col0 ..; this lane's row packed in h, columns in pairs) for a C
// whose rows TMA cannot describe: the rows go through the warp's staging
// buffer `sb` (32 x 128 bytes, 128B-swizzled) and are written row by row,
// lane l owning columns 2l and 2l + 1, skipping rows >= M and columns >= N.
__device__ __forceinline__ void store_rows_predicated(uint32_t sb, const uint32_t (&h)[32],
                                                      uint16_t *C, int64_t M, int64_t N,
                                                      int64_t row0, int64_t col0, int lane) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        st_shared_v4(sb + sw128_offset(lane, j), h[4 * j], h[4 * j + 1], h[4 * j + 2],
                     h[4 * j + 3]);
    __syncwarp();
    const int64_t col = col0 + 2 * lane;
    for (int rr = 0; rr < 32; ++rr) {
        const int64_t row = row0 + rr;
        if (row >= M)
            break;
        const uint32_t w = ld_shared_b32(sb + rr * 128u + ((((uint32_t)lane >> 2) ^ (rr & 7u)) << 4) +
                                         ((uint32_t)lane & 3u) * 4u);
        uint16_t *dst = C + row * N + col;
        if (col + 1 < N && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
            *reinterpret_cast<uint32_t *>(dst) = w;
        } else {
            if (col < N)
                dst[0] = (uint16_t)(w & 0xffffu);
            if (col + 1 < N)
                dst[1] = (uint16_t)(w >> 16);
        }
    }
    __syncwarp();
}

// Keep the first `nvalid` fp16 values of an 8-value chunk, zero the rest.
__device__ __forceinline__ uint32_t keep_pair(uint32_t w, int nvalid, int e) {
    return e >= nvalid ? 0u : (e + 1 >= nvalid ? (w & 0xffffu) : w);
}

__device__ __forceinline__ uint4 keep_first(uint4 v, int nvalid) {
    if (nvalid >= 8)
        return v;
    return make_uint4(keep_pair(v.x, nvalid, 0), keep_pair(v.y, nvalid, 2),
                      keep_pair(v.z, nvalid, 4), keep_pair(v.w, nvalid, 6));
}

// tcgen05.ld of 32 / 16 columns fused with its wait, so that no use of the
// destination registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld_x32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x16_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// ================================================================== fused kernel

namespace fused {

constexpr int BM = 128;            // UMMA M: TMEM lanes = output rows
constexpr int BK = 64;             // one 128-byte swizzle row of fp16
constexpr int UK = 16;             // K of one tcgen05.mma kind::f16
constexpr uint32_t kATile = BM * BK * 2;    // 16 KB, K-major, 128 rows x 128 B
constexpr uint32_t kBSlab = BK * 64 * 2;    // 8 KB: 64 k-rows x 64 n (128 B)
constexpr uint32_t kEpiBuf = 32 * 128;      // 32 rows x 64 fp16, swizzled
constexpr int kEpiWarps = 4;

// Per tile width BN (UMMA N = TMEM columns per accumulator): 256 or 128.
// The TMA kernels' ring gets as many stages as fit beside 32 KB of epilogue
// staging (two buffers per epilogue warp).  The predicated-load kernel
// (kTma false, BN = 128) keeps two operand stages and, before them, a ring of
// kRawStages raw stages: the aligned 16-byte blocks of each row segment as
// TMA brings them (A: 128 rows of 9 blocks, B: 64 k-rows of 17 blocks,
// grouped by row residue modulo 8), which its producers shift into the
// operand layout; its epilogue stores from one staging buffer per warp.
template <int kBN, bool kTma = true>
struct Tile {
    static constexpr int BN = kBN;
    static constexpr uint32_t kBTile = BK * BN * 2;          // BN / 64 slabs, MN-major
    static constexpr int kStages = kTma ? (kBN >= 256 ? 4 : 6) : 2;
    static constexpr int kRawStages = kTma ? 0 : 3;
    static constexpr int kEpiBufs = kTma ? 2 : 1;            // staging buffers per epilogue warp
    static constexpr uint32_t kRawRowA = (BK / 8 + 1) * 16;  // 144 B
    static constexpr uint32_t kRawRowB = (BN / 8 + 1) * 16;  // 272 B at BN = 128
    static constexpr uint32_t kRawB = BM * kRawRowA;         // B rows follow the A rows
    static constexpr uint32_t kRawStage = kRawB + BK * kRawRowB;
    static constexpr uint32_t kTmemCols = 2 * BN;            // double-buffered accumulator
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kOffA + kStages * kATile;
    static constexpr uint32_t kOffRaw = kOffB + kStages * kBTile;
    static constexpr uint32_t kOffEpi = kOffRaw + kRawStages * kRawStage;
    static constexpr uint32_t kOffBar = kOffEpi + kEpiWarps * kEpiBufs * kEpiBuf;
    static constexpr uint32_t kNumBars = 2 * kStages + 4 + 1 + 8 * kRawStages;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemUsed = kOffMisc + 16;
    static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
    // A: K-major (bit 15 = 0); B: N-major (bit 16 = 1); M = 128, N = BN.
    static constexpr uint32_t kIdesc = make_idesc_f16_f32(BM, BN, 0, 1);
    static_assert(kOffEpi % 1024 == 0 && kSmemBytes <= 232448, "shared memory layout");
};

struct Params {
    const uint16_t *A;
    const uint16_t *B;
    uint16_t *C;
    int M, N, K;
    int num_kb;
    int64_t m_tiles, n_tiles, num_tiles;
    int panel;
    int drop_arrive;
    uint64_t wait_limit_ns;
    // Stream-K schedule ("TileLang tutorial", chapter "Persistent kernel":
    // split-K / stream-K remove the partial last wave).  Tiles [0, dp_tiles)
    // run data-parallel: CTA c takes tiles c, c + G, ...  The k blocks of the
    // remaining tiles are laid end to end and cut into G equal contiguous
    // ranges, one per CTA, so every CTA gets the same amount of MMA work.  A
    // tile cut between CTA c (its k head: the first k blocks, at the end of
    // c's range) and CTA c + 1 (its k tail, at the start of c + 1's range) is
    // finished by whichever of the two gets there second (see sk_exchange):
    // no CTA ever waits for another.  With fewer tiles than CTAs (dp_tiles
    // 0, ranges shorter than a tile) a tile can be cut more than once; its
    // cuts are then settled from right to left (see the epilogue), so the
    // tile is always summed as p0 + (p1 + (p2 + ...)) over its pieces.
    // dp_tiles equal to num_tiles means no stream-K part.
    int64_t dp_tiles;
    float *sk_part;        // [G] k-tail slots of BM x BN fp32, [BN/4][BM][4] each
    float *sk_head;        // [G] k-head slots, same layout
    uint32_t *sk_flags;    // [G][4]: the state of each cut, one word per epilogue warp
    uint32_t epoch;        // nonzero, below 2^30, distinct per call
    int sk_mode;           // test hook: 0 normal; 1 heads always publish; 2 also delay
                           // tails; 3 heads always publish, delayed
};

// Tensor maps of the predicated-load kernel: for each residue a modulo 8, the
// rows a, a + 8, a + 16, ... of A (and of B) as a 2-D tensor whose base is the
// first such row's start rounded down to 16 bytes and whose row stride is 8
// rows (16 * cols bytes, a multiple of 16 whatever cols is).  Element x of
// such a tensor row is element x - off / 2 of the matrix row (off = the byte
// offset of the row start inside its 16-byte block), so a box starting at
// x = k0 brings the aligned blocks that hold elements k0 .. of every row,
// with the k (or n) tail and the rows past the end zero-filled.
struct RowMaps {
    CUtensorMap a[8];      // box: 72 elements (144 B) x 16 rows
    CUtensorMap b[8];      // box: 136 elements (272 B) x 8 rows
};
struct NoMaps {};
template <bool kTma>
using MapsFor = typename std::conditional<kTma, NoMaps, RowMaps>::type;

enum ItemKind : int { kItemFull = 0, kItemPieceOut = 1, kItemPieceIn = 2, kItemPieceMid = 3 };

// Stream-K schedule over `num_tiles` tiles of `num_kb` k blocks run by G
// workers (CTAs, or CTA pairs): tiles [0, dp_tiles) data-parallel, worker c
// taking c, c + G, ...; the k blocks of the other tiles laid end to end and
// cut into G equal contiguous ranges.
struct SkShape {
    int64_t num_tiles, dp_tiles, num_kb;
};

// Number of work items of worker c (data-parallel tiles, then pieces).
__device__ __forceinline__ int64_t sk_num_items(const SkShape &g, int64_t c, int64_t G) {
    const int64_t ndp = c < g.dp_tiles ? (g.dp_tiles - 1 - c) / G + 1 : 0;
    const int64_t W = (g.num_tiles - g.dp_tiles) * g.num_kb;
    const int64_t s = c * W / G, e = (c + 1) * W / G;
    if (e <= s)
        return ndp;
    return ndp + (e - 1) / g.num_kb - s / g.num_kb + 1;
}

// Item i of worker c: tile id, k-block range [kb0, kb1) and kind.  A piece
// that starts inside its tile is the tile's k tail (kItemPieceOut); one that
// stops inside is its k head (kItemPieceIn); one that does both
// (kItemPieceMid) lies strictly inside a tile, which happens only when the
// ranges are shorter than a tile (fewer tiles than workers).  The CTA-pair
// kernel's schedules always have ranges of at least one tile.
__device__ __forceinline__ void sk_item_at(const SkShape &g, int64_t c, int64_t G, int64_t i,
                                           int64_t &tile, int &kb0, int &kb1, int &kind) {
    const int64_t ndp = c < g.dp_tiles ? (g.dp_tiles - 1 - c) / G + 1 : 0;
    if (i < ndp) {
        tile = c + i * G;
        kb0 = 0;
        kb1 = (int)g.num_kb;
        kind = kItemFull;
        return;
    }
    const int64_t W = (g.num_tiles - g.dp_tiles) * g.num_kb;
    const int64_t s = c * W / G, e = (c + 1) * W / G;
    const int64_t t = s / g.num_kb + (i - ndp);
    const int64_t lo = t * g.num_kb;
    kb0 = (int)((s > lo ? s : lo) - lo);
    kb1 = (int)((e < lo + g.num_kb ? e : lo + g.num_kb) - lo);
    tile = g.dp_tiles + t;
    kind = kb0 > 0 ? (kb1 < g.num_kb ? kItemPieceMid : kItemPieceOut)
                   : (kb1 < g.num_kb ? kItemPieceIn : kItemFull);
}

__device__ __forceinline__ int64_t num_items(const Params &p, int64_t c, int64_t G) {
    return sk_num_items(SkShape{p.num_tiles, p.dp_tiles, p.num_kb}, c, G);
}

__device__ __forceinline__ void item_at(const Params &p, int64_t c, int64_t G, int64_t i,
                                        int64_t &tile, int &kb0, int &kb1, int &kind) {
    sk_item_at(SkShape{p.num_tiles, p.dp_tiles, p.num_kb}, c, G, i, tile, kb0, kb1, kind);
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Stream-K fix-up of a tile cut between two workers, wait-free.  The state
// word of the cut (one per epilogue warp) is tagged with the call's epoch:
// sk_tail_tag when the k tail's fp32 piece is published, sk_head_tag when the
// k head's is.  Each side publishes its piece only if it may be first, then
// swaps its tag into the word; the side whose swap returns the other's tag
// came second and finishes the tile (adds the published piece to its own and
// stores C).  Exactly one side finishes, neither waits, so the kernels need
// no co-residency guarantee.  The sum is own + other in fp32, which is the
// same number whichever side adds (fp32 addition is commutative).
__device__ __forceinline__ uint32_t sk_tail_tag(uint32_t epoch) { return epoch * 4u + 1u; }
__device__ __forceinline__ uint32_t sk_head_tag(uint32_t epoch) { return epoch * 4u + 2u; }

// Warp-uniform read of a cut's state: lane 0 loads it with acquire, the warp
// synchronises, and every lane fences, so every lane's later loads of the
// other side's piece come after the load that saw its tag.
__device__ __forceinline__ uint32_t sk_peek(const uint32_t *state, int lane) {
    uint32_t v = 0;
    if (lane == 0)
        v = ld_acquire_gpu(state);
    v = __shfl_sync(0xffffffffu, v, 0);
    __syncwarp();
    __threadfence();
    return v;
}

// Warp-uniform swap of `tag` into a cut's state after this warp's piece
// stores (each lane fences its stores, the warp synchronises, lane 0 fences
// again -- fences are cumulative -- and swaps); returns the previous state,
// with the same ordering as sk_peek for the loads that follow.
__device__ __forceinline__ uint32_t sk_exchange(uint32_t *state, uint32_t tag, int lane) {
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) {
        __threadfence();
        old = atomicExch(state, tag);
        __threadfence();
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    __syncwarp();
    __threadfence();
    return old;
}

// r[j] += column col0 + j of this lane's row of a published piece.
__device__ __forceinline__ void add_slot32(uint32_t (&r)[32], const float *slot, int row,
                                           int col0) {
    const float4 *s = reinterpret_cast<const float4 *>(slot) + (size_t)(col0 / 4) * 128 + row;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x = __ldcg(s + (size_t)i * 128);
        r[4 * i] = __float_as_uint(__uint_as_float(r[4 * i]) + x.x);
        r[4 * i + 1] = __float_as_uint(__uint_as_float(r[4 * i + 1]) + x.y);
        r[4 * i + 2] = __float_as_uint(__uint_as_float(r[4 * i + 2]) + x.z);
        r[4 * i + 3] = __float_as_uint(__uint_as_float(r[4 * i + 3]) + x.w);
    }
}

// r[j] = column col0 + j of this lane's row of a published piece.
__device__ __forceinline__ void load_slot32(uint32_t (&r)[32], const float *slot, int row,
                                            int col0) {
    const float4 *s = reinterpret_cast<const float4 *>(slot) + (size_t)(col0 / 4) * 128 + row;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x = __ldcg(s + (size_t)i * 128);
        r[4 * i] = __float_as_uint(x.x);
        r[4 * i + 1] = __float_as_uint(x.y);
        r[4 * i + 2] = __float_as_uint(x.z);
        r[4 * i + 3] = __float_as_uint(x.w);
    }
}

// Test hook: keep one side of a cut from publishing for about `ns` (bounded
// by the global timer), so the other side of the exchange runs first.
__device__ __forceinline__ void sk_test_delay(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns)
        __nanosleep(1000);
}

// r[j] += the 32 fp32 columns at TMEM address taddr (this lane's row).
__device__ __forceinline__ void add_tmem(uint32_t (&r)[32], uint32_t taddr) {
    uint32_t o[32];
    tmem_ld_x32_sync(taddr, o);
#pragma unroll
    for (int j = 0; j < 32; ++j)
        r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(o[j]));
}

// A stream-K piece of 128 rows x kCols fp32 columns is kept in its slot as
// [kCols / 4][128][4]: the four consecutive columns a lane holds for its row
// are one 16-byte vector, and the 32 rows of a warp are 512 contiguous bytes.
//
// piece_store32: store this lane's row, columns col0 .. col0 + 31 (r from a
// 32-column TMEM load), at L2 (the reader is another SM).
__device__ __forceinline__ void piece_store32(float *slot, int row, int col0,
                                              const uint32_t (&r)[32]) {
    float4 *d = reinterpret_cast<float4 *>(slot) + (size_t)(col0 / 4) * 128 + row;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        __stcg(d + (size_t)i * 128,
               make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                           __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
}

// piece_to_tmem: copy this lane's row of a whole kCols-column piece into TMEM
// columns taddr .. taddr + kCols - 1.  Four 32-column chunks (32 vector loads)
// are in flight at once, so the copy costs kCols / 128 L2 round trips.
template <int kCols>
__device__ __forceinline__ void piece_to_tmem(const float *slot, int row, uint32_t taddr) {
    constexpr int kBatch = kCols / 32 < 4 ? kCols / 32 : 4;
    const float4 *src = reinterpret_cast<const float4 *>(slot) + row;
#pragma unroll 1
    for (int c0 = 0; c0 < kCols / 32; c0 += kBatch) {
        uint32_t v[kBatch][32];
#pragma unroll
        for (int cc = 0; cc < kBatch; ++cc) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 x = __ldcg(src + (size_t)((c0 + cc) * 8 + i) * 128);
                v[cc][4 * i] = __float_as_uint(x.x);
                v[cc][4 * i + 1] = __float_as_uint(x.y);
                v[cc][4 * i + 2] = __float_as_uint(x.z);
                v[cc][4 * i + 3] = __float_as_uint(x.w);
            }
        }
#pragma unroll
        for (int cc = 0; cc < kBatch; ++cc)
            tmem_st_x32(taddr + 32 * (c0 + cc), v[cc]);
    }
    tmem_st_wait();
}

template <bool kTma>
struct Roles {
    static constexpr int kLoadWarps = kTma ? 1 : 8;
    static constexpr int kMmaWarp = kLoadWarps;
    static constexpr int kEpiWarp0 = kLoadWarps + 1;
    static constexpr int kThreads = 32 * (kLoadWarps + 1 + kEpiWarps);
};

// kTma: operands by TMA (else the predicated-load producer); kTmaStore: C by
// TMA (else predicated stores, for a C whose rows TMA cannot describe).
template <bool kTma, int kBN, bool kTmaStore = kTma>
__global__ void __launch_bounds__(Roles<kTma>::kThreads, 1)
    gemm_relu_fused_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const Params p,
                           const __grid_constant__ MapsFor<kTma> rm) {
    using R = Roles<kTma>;
    using T = Tile<kBN, kTma>;
    constexpr int BN = T::BN;
    constexpr int kStages = T::kStages;
    constexpr uint32_t kBTile = T::kBTile, kTmemCols = T::kTmemCols, kIdesc = T::kIdesc;
    constexpr uint32_t kOffA = T::kOffA, kOffB = T::kOffB, kOffEpi = T::kOffEpi;
    constexpr uint32_t kOffBar = T::kOffBar, kOffMisc = T::kOffMisc;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + kOffBar;
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (kStages + s); };
    auto accf_bar = [&](uint32_t b) { return bar0 + 8u * (2 * kStages + b); };
    auto acce_bar = [&](uint32_t b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kOffMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), kTma ? 1u : (uint32_t)R::kLoadWarps);
            mbar_init(empty_bar(s), 1u);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1u);
            mbar_init(acce_bar(b), (uint32_t)kEpiWarps);
        }
        mbar_init(drain_bar, 1u);
        for (int b = 0; b < 8 * T::kRawStages; ++b)
            mbar_init(drain_bar + 8u * (1u + (uint32_t)b), 1u);
        *abort_flag = 0u;
        fence_mbar_init();
        pdl_launch_dependents();
    }
    if (kTma && warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        if (kTmaStore)
            tma_prefetch_map(&tmC);
    }
    if (warp == R::kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    pdl_wait_primary();  // the previous grid of the stream has completed

    if (warp < R::kLoadWarps) {
        // ============================================================ producer
        if constexpr (kTma) {
            if (lane == 0) {
                uint32_t stage = 0, phase = 0, issued = 0, parity = 0;
                bool ok = true;
                const int64_t items = num_items(p, blockIdx.x, gridDim.x);
                for (int64_t it = 0; ok && it < items; ++it) {
                    int64_t t, mb, nb;
                    int kb0, kb1, kind;
                    item_at(p, blockIdx.x, gridDim.x, it, t, kb0, kb1, kind);
                    tile_coord(t, p.m_tiles, p.n_tiles, p.panel, mb, nb);
                    const int m0 = (int)(mb * BM), n0 = (int)(nb * BN);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_limit_ns, abort_flag,
                                          kSiteProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        const bool drop = p.drop_arrive && blockIdx.x == 0 && it == 0 && kb == kb0;
                        if (!drop) {
                            const uint32_t fb = full_bar(stage);
                            mbar_arrive_expect_tx(fb, kATile + kBTile);
                            tma_load_2d(&tmA, base + kOffA + stage * kATile, fb, kb * BK, m0);
                            const uint32_t bdst = base + kOffB + stage * kBTile;
#pragma unroll
                            for (int j = 0; j < BN / 64; ++j)
                                tma_load_2d(&tmB, bdst + j * kBSlab, fb, n0 + 64 * j, kb * BK);
                            issued |= 1u << stage;
                            parity = (parity & ~(1u << stage)) | (phase << stage);
                        }
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                // Every copy issued must have landed before the CTA may exit.
                for (uint32_t s = 0; s < kStages; ++s)
                    if (issued & (1u << s))
                        wait_drain(full_bar(s), (parity >> s) & 1u, p.wait_limit_ns, abort_flag);
            }
        } else {
            // Predicated loads for operands TMA cannot describe (see window16
            // and RowMaps).  Eight warps; warp w handles the rows of residue w
            // modulo 8 of every stage: A rows w + 8i (i < 16), B k-rows w + 8i
            // (i < 8).  Its lane 0 loads them into its part of a raw slot with
            // two TMA boxes, kRawStages - 1 stages ahead; once they have
            // landed, the warp shifts them into the operand stage: A as four
            // ops of four rows x 8 lanes (a row's 64 k = 128 bytes), B as four
            // ops of two rows x 16 lanes (a k-row's 128 n = 256 bytes, both
            // 64-wide slabs).  Each lane reads the raw blocks c and c + 1 of
            // its row.  A warp reads only the raw rows its own lane 0 loaded.
            static_assert(BN == 128 && R::kLoadWarps == 8,
                          "the predicated-load producer is laid out for 128 x 128 tiles, 8 warps");
            constexpr int kRaw = T::kRawStages;
            constexpr uint32_t kRawRowA = T::kRawRowA, kRawRowB = T::kRawRowB;
            constexpr uint32_t kResA = 16 * kRawRowA;     // one residue's A rows: 2304 B
            constexpr uint32_t kResB = 8 * kRawRowB;      // one residue's B k-rows: 2176 B
            const int g8 = lane >> 3, c8 = lane & 7;
            const int g16 = lane >> 4, c16 = lane & 15;
            const bool has_a = p.M > warp, has_b = p.K > warp;   // residue has rows at all
            const uint32_t tx = (has_a ? kResA : 0u) + (has_b ? kResB : 0u);
            const Shift fa = make_shift((uint32_t)((reinterpret_cast<uintptr_t>(p.A) +
                                                    2ull * (uint64_t)warp * (uint64_t)p.K) & 15u));
            const Shift fb = make_shift((uint32_t)((reinterpret_cast<uintptr_t>(p.B) +
                                                    2ull * (uint64_t)warp * (uint64_t)p.N) & 15u));
            const CUtensorMap *map_a = &rm.a[warp];
            const CUtensorMap *map_b = &rm.b[warp];
            if (lane == 0) {
                if (has_a)
                    tma_prefetch_map(map_a);
                if (has_b)
                    tma_prefetch_map(map_b);
            }
            auto raw_bar = [&](uint32_t j) { return drain_bar + 8u * (1u + (uint32_t)warp * kRaw + j); };
            const int64_t items = num_items(p, blockIdx.x, gridDim.x);
            struct Cursor {
                int64_t it;
                int m0, n0, kb, kb0, kb1;
            };
            auto open = [&](Cursor &cu, int64_t i) {
                int64_t t, mb, nb;
                int kind;
                item_at(p, blockIdx.x, gridDim.x, i, t, cu.kb0, cu.kb1, kind);
                tile_coord(t, p.m_tiles, p.n_tiles, p.panel, mb, nb);
                cu.it = i;
                cu.kb = cu.kb0;
                cu.m0 = (int)(mb * BM);
                cu.n0 = (int)(nb * BN);
            };
            auto advance = [&](Cursor &cu) -> bool {
                if (++cu.kb < cu.kb1)
                    return true;
                if (cu.it + 1 >= items)
                    return false;
                open(cu, cu.it + 1);
                return true;
            };
            // stage `cu`'s rows of this residue into raw slot j
            auto issue = [&](const Cursor &cu, uint32_t j) {
                if (lane != 0)
                    return;
                const uint32_t rb = raw_bar(j);
                const uint32_t raw = base + T::kOffRaw + j * T::kRawStage;
                if (tx == 0u) {
                    mbar_arrive(rb);
                    return;
                }
                mbar_arrive_expect_tx(rb, tx);
                if (has_a)
                    tma_load_2d(map_a, raw + (uint32_t)warp * kResA, rb, cu.kb * BK, cu.m0 / 8);
                if (has_b)
                    tma_load_2d(map_b, raw + T::kRawB + (uint32_t)warp * kResB, rb, cu.n0,
                                cu.kb * (BK / 8));
            };
            // raw slot j -> operand stage `stage`: all sixteen block reads
            // first, then the shifts and stores.  (Reading one block and
            // taking the next from the neighbour lane with shuffles measured
            // slower: the shuffles share the shared-memory pipe.)
            auto fix_stage = [&](uint32_t j, uint32_t stage) {
                const uint32_t raw = base + T::kOffRaw + j * T::kRawStage;
                const uint32_t adst = base + kOffA + stage * kATile;
                const uint32_t bdst = base + kOffB + stage * kBTile;
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                uint4 v[8][2];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t sa = raw + (uint32_t)warp * kResA +
                                        (uint32_t)(4 * t + g8) * kRawRowA + 16u * (uint32_t)c8;
                    v[t][0] = ld_shared_v4(sa);
                    v[t][1] = ld_shared_v4(sa + 16u);
                    const uint32_t sb = raw + T::kRawB + (uint32_t)warp * kResB +
                                        (uint32_t)(2 * t + g16) * kRawRowB + 16u * (uint32_t)c16;
                    v[4 + t][0] = ld_shared_v4(sb);
                    v[4 + t][1] = ld_shared_v4(sb + 16u);
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint4 o = has_a ? window16(v[t][0], v[t][1], fa) : z;
                    st_shared_v4(adst + sw128_offset((uint32_t)(warp + 8 * (4 * t + g8)), (uint32_t)c8),
                                 o.x, o.y, o.z, o.w);
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint4 o = has_b ? window16(v[4 + t][0], v[4 + t][1], fb) : z;
                    st_shared_v4(bdst + (uint32_t)(c16 >> 3) * kBSlab +
                                     sw128_offset((uint32_t)(warp + 8 * (2 * t + g16)),
                                                  (uint32_t)(c16 & 7)),
                                 o.x, o.y, o.z, o.w);
                }
            };
            Cursor cp{}, fx{};
            bool cp_more = items > 0, fx_more = items > 0;
            if (cp_more) {
                open(cp, 0);
                fx = cp;
            }
            uint32_t issued = 0, fixed = 0;      // stages loaded / shifted by this warp
            for (int i = 0; i < kRaw - 1 && cp_more; ++i) {
                issue(cp, issued % kRaw);
                ++issued;
                cp_more = advance(cp);
            }
            uint32_t stage = 0, phase = 0;
            while (fx_more) {
                // the next load goes into the slot shifted last (read complete:
                // ordered by that stage's proxy fence and __syncwarp)
                if (cp_more) {
                    issue(cp, issued % kRaw);
                    ++issued;
                    cp_more = advance(cp);
                }
                const uint32_t j = fixed % kRaw;
                bool ok = true;
                // (both usually complete already: poll without the suspend
                // hint, which measured faster here)
                if (lane == 0)
                    ok = wait_bounded_eager(raw_bar(j), (fixed / kRaw) & 1u, p.wait_limit_ns,
                                            abort_flag, kSiteProducerEmpty) &&
                         wait_bounded_eager(empty_bar(stage), phase ^ 1u, p.wait_limit_ns,
                                            abort_flag, kSiteProducerEmpty);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0))
                    break;
                fix_stage(j, stage);
                // every lane's stores made visible to the tensor core (and its
                // raw reads ordered before the next TMA write of the slot),
                // then one arrival per warp
                fence_proxy_async_smem();
                __syncwarp();
                const bool drop = p.drop_arrive && blockIdx.x == 0 && fx.it == 0 && fx.kb == fx.kb0;
                if (lane == 0 && !drop)
                    mbar_arrive(full_bar(stage));
                ++fixed;
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                fx_more = advance(fx);
            }
            // loads still in flight after an abort must land before the CTA exits
            if (lane == 0)
                for (uint32_t q = fixed; q < issued; ++q)
                    wait_drain(raw_bar(q % kRaw), (q / kRaw) & 1u, p.wait_limit_ns, abort_flag);
        }
    } else if (warp == R::kMmaWarp) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            const int64_t items = num_items(p, blockIdx.x, gridDim.x);
            for (int64_t i = 0; ok && i < items; ++i) {
                int64_t t;
                int kb0, kb1, kind;
                item_at(p, blockIdx.x, gridDim.x, i, t, kb0, kb1, kind);
                const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
                if (!wait_bounded(acce_bar(buf), use ^ 1u, p.wait_limit_ns, abort_flag,
                                  kSiteMmaAccEmpty))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + buf * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, p.wait_limit_ns, abort_flag,
                                      kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a = base + kOffA + stage * kATile;
                    const uint32_t b = base + kOffB + stage * kBTile;
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk) {
                        // A (K-major): the next 16 k are 32 bytes further
                        // along each swizzled row; 8-row groups 1024 B apart.
                        const uint64_t adesc = make_sdesc_sw128(a + kk * (UK * 2), 16, 1024);
                        // B (N-major): the next 16 k are 16 rows of 128 B
                        // further; 64-wide N slabs kBSlab apart (LBO), 8-row
                        // k groups 1024 B apart (SBO).
                        const uint64_t bdesc = make_sdesc_sw128(b + kk * (UK * 128), kBSlab, 1024);
                        umma_f16(d, adesc, bdesc, kIdesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(empty_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit(accf_bar(buf));
            }
            // All MMAs of this thread complete before TMEM can be released.
            umma_commit(drain_bar);
            wait_drain(drain_bar, 0u, p.wait_limit_ns, abort_flag);
        }
    } else {
        // ============================================================ epilogue
        const int ew = warp - R::kEpiWarp0;     // staging buffer owner 0..3
        const int q = warp & 3;                 // TMEM lanes 32q .. 32q+31
        const int row_in_tile = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t stage_base = base + kOffEpi + (uint32_t)ew * T::kEpiBufs * kEpiBuf;
        uint32_t nstores = 0;
        const int64_t items = num_items(p, blockIdx.x, gridDim.x);
        // Stream-K.  Cut k (0 < k < G) sits at position k * W / G of the
        // stream-K k blocks; its state word is sk_flags[k][q], the pieces on
        // its two sides go to sk_part[k] (everything of the tile right of the
        // cut) and sk_head[k - 1] (CTA k - 1's own piece, left of the cut).
        // This CTA's first stream-K item starts at cut c = blockIdx.x and its
        // last ends at cut c + 1.  When the k head is the last item and the
        // next CTA's k tail is already published by the time the item before
        // it has been read, the tail is copied into the other TMEM buffer (not
        // used again) while the MMA works on the head, and the head's epilogue
        // adds the two buffers; otherwise the two sides meet through
        // sk_exchange.
        int64_t last_t = 0;
        int last_kb0 = 0, last_kb1 = 0, last_kind = kItemFull;
        if (items > 0)
            item_at(p, blockIdx.x, gridDim.x, items - 1, last_t, last_kb0, last_kb1, last_kind);
        // (not in the predicated-load kernel: its 13 warps leave 128
        // registers a thread, which the pre-load's 128 in-flight values
        // would overflow)
        const bool head_last = kTma && last_kind == kItemPieceIn;
        const uint32_t partner_buf = tmem_base + lane_base + (uint32_t)((items - 2) & 1) * BN;
        const int64_t sk_w = (p.num_tiles - p.dp_tiles) * (int64_t)p.num_kb;
        constexpr size_t kSlot = (size_t)BN * BM;
        auto cut_state = [&](int64_t k) { return p.sk_flags + k * 4 + q; };
        uint32_t *const head_cut = cut_state((int64_t)blockIdx.x + 1);   // this CTA's k head
        const float *const next_tail = p.sk_part + (size_t)(blockIdx.x + 1) * kSlot;
        bool preloaded = false;
        auto try_preload = [&]() {
            if (p.sk_mode != 0 || sk_peek(head_cut, lane) != sk_tail_tag(p.epoch))
                return;
            piece_to_tmem<BN>(next_tail, row_in_tile, partner_buf);
            __syncwarp();
            if (lane == 0)
                *head_cut = 0u;  // consumed
            preloaded = true;
        };
        // A sum of pieces in fp32: the TMEM accumulator `acc` (or the
        // published piece `from`, when set) plus either the TMEM partner
        // buffer (when `partner`) or the published piece `add` (when set).
        // sum32: columns col0 .. col0 + 31 of this lane's row.
        auto sum32 = [&](uint32_t acc, const float *from, bool partner, const float *add,
                         int col0, uint32_t (&r)[32]) {
            if (from)
                load_slot32(r, from, row_in_tile, col0);
            else
                tmem_ld_x32_sync(acc + (uint32_t)col0, r);
            if (partner)
                add_tmem(r, partner_buf + (uint32_t)col0);
            else if (add)
                add_slot32(r, add, row_in_tile, col0);
        };
        // Stores tile t from a sum of pieces (as in sum32) as ReLU'd fp16.
        auto store_tile = [&](int64_t t, uint32_t acc, const float *from, bool partner,
                              const float *add) {
            int64_t mb, nb;
            tile_coord(t, p.m_tiles, p.n_tiles, p.panel, mb, nb);
            const int64_t row0 = mb * BM + 32 * q;
            const int64_t n0 = nb * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 64; ++c) {
                const int64_t col0 = n0 + 64 * c;
                if (row0 >= p.M || col0 >= p.N)
                    continue;  // warp-uniform: nothing of this chunk is in C
                uint32_t r[32], h[32];
                sum32(acc, from, partner, add, 64 * c, r);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    h[j] = relu_pack_half2(r[2 * j], r[2 * j + 1]);
                sum32(acc, from, partner, add, 64 * c + 32, r);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    h[16 + j] = relu_pack_half2(r[2 * j], r[2 * j + 1]);
                if constexpr (kTmaStore) {
                    const uint32_t sb = stage_base + (nstores & 1u) * kEpiBuf;
                    // the store issued two chunks ago from this buffer must
                    // have finished reading it
                    if (lane == 0)
                        bulk_wait_group_read<1>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(sb + sw128_offset(lane, j), h[4 * j], h[4 * j + 1],
                                     h[4 * j + 2], h[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, sb, (int32_t)col0, (int32_t)row0);
                        bulk_commit_group();
                    }
                    ++nstores;
                } else {
                    store_rows_predicated(stage_base, h, p.C, p.M, p.N, row0, col0, lane);
                }
            }
        };
        // Publishes this lane's row of a sum of pieces (as in sum32) into `slot`.
        auto publish = [&](float *slot, uint32_t acc, const float *from, const float *add) {
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                sum32(acc, from, false, add, 32 * c, r);
                piece_store32(slot, row_in_tile, 32 * c, r);
            }
        };
        for (int64_t i = 0; i < items; ++i) {
            int64_t t;
            int kb0, kb1, kind;
            item_at(p, blockIdx.x, gridDim.x, i, t, kb0, kb1, kind);
            const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
            // (the predicated-load kernel's producers share the schedulers
            // with these warps: poll slowly there)
            const bool ok = kTma ? wait_bounded(accf_bar(buf), use, p.wait_limit_ns, abort_flag,
                                                kSiteEpiAccFull)
                                 : wait_bounded_sleep(accf_bar(buf), use, p.wait_limit_ns,
                                                      abort_flag, kSiteEpiAccFull, 256);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after_sync();
            const uint32_t acc = tmem_base + lane_base + buf * BN;
            // the sum this warp holds of the tile: acc (or `from`) + partner + add
            const float *from = nullptr, *add = nullptr;
            bool partner = false;
            bool holds = true;  // this warp still holds part of the tile's sum
            // (stream-K schedules run on the TMA kernels only: the host plans
            // none for the predicated-load kernel, whose items are all whole)
            if (kTma && (kind == kItemPieceIn || kind == kItemPieceMid)) {
                // The cut at the piece's end first (this CTA is its left side):
                // add the next CTA's published right part if it is there; else
                // publish the piece, and go on only if the right part arrived
                // meanwhile (otherwise its owner goes on with this piece).
                if (p.sk_mode == 3)
                    sk_test_delay(200000);
                if (preloaded) {
                    partner = true;
                } else if (p.sk_mode == 0 && sk_peek(head_cut, lane) == sk_tail_tag(p.epoch)) {
                    add = next_tail;
                } else {
                    publish(p.sk_head + (size_t)blockIdx.x * kSlot, acc, nullptr, nullptr);
                    if (sk_exchange(head_cut, sk_head_tag(p.epoch), lane) == sk_tail_tag(p.epoch))
                        add = next_tail;
                    else
                        holds = false;
                }
                if (add) {
                    __syncwarp();
                    if (lane == 0)
                        *head_cut = 0u;  // consumed (nobody touches it again in this call)
                }
            }
            // Then the cuts to the left, while the sum held starts inside the
            // tile: publish it as the right part of cut k; if cut k's left
            // piece (CTA k - 1's) was published first, add it, and the sum now
            // starts where CTA k - 1's range does.
            int64_t k = blockIdx.x;
            bool inside = kTma && kb0 > 0;
            if (holds && inside && p.sk_mode == 2)
                sk_test_delay(200000);
            const int64_t tile_lo = (t - p.dp_tiles) * (int64_t)p.num_kb;
            while (holds && inside) {
                float *const slot = p.sk_part + (size_t)k * kSlot;
                publish(slot, acc, from, add);
                if (sk_exchange(cut_state(k), sk_tail_tag(p.epoch), lane) != sk_head_tag(p.epoch)) {
                    holds = false;  // CTA k - 1 finishes the cut
                    break;
                }
                __syncwarp();
                if (lane == 0)
                    *cut_state(k) = 0u;  // consumed
                from = slot;
                add = p.sk_head + (size_t)(k - 1) * kSlot;
                inside = (k - 1) * sk_w / (int64_t)gridDim.x > tile_lo;
                --k;
            }
            if (holds)
                store_tile(t, acc, from, partner, add);
            // accumulator buffer fully read: hand it back to the MMA warp
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce_bar(buf));
            if (head_last && items >= 2 && i == items - 2)
                try_preload();
        }
        if constexpr (kTmaStore) {
            if (lane == 0)
                bulk_wait_group<0>();
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == R::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace fused


}  // namespace gemmrelu
