// gemm_relu_splitk.cuh -- split-K fused GEMM + ReLU for skinny (memory-bound)
// shapes.
//
// The split-K scheme of "TileLang 编程基本知识点" section 5.1 cuts the K range
// into S pieces computed by different CTAs; each piece only offsets K.  The
// page adds the fp32 partials with atomics into a pre-zeroed C, and notes
// that for reproducible results the partials should instead be kept and
// reduced in a separate step.  Here the S raw fp32 partials (no ReLU) are
// always summed in the fixed order 0, 1, ..., S-1 starting from 0, then the
// ReLU and the fp16 cast follow, in one of two forms:
//
//   CTA-pair form (gemm_relu_splitk_kernel<BMS, true>): a cluster of two
//     CTAs computes all pieces of a tile, half each, one TMEM accumulator
//     per piece; the first CTA's running sum moves to the second through
//     distributed shared memory and the second finishes the sum and stores
//     C.  One kernel, no workspace.
//   two-stage form: gemm_relu_splitk_kernel<BMS, false> writes every
//     piece's partial to part[s][m][n]; gemm_relu_splitk_reduce_kernel, a
//     programmatic dependent launch, sums them and stores C.
//
// Both compute C^T = B^T . A^T: the MMA's M side (128 TMEM lanes) runs over
// N and its narrow N side (BMS columns) over M, so M = 16 costs a 128 x 16
// MMA instead of a mostly empty 128-row tile.  UMMA A operand = a B tile,
// N-major; UMMA B operand = an A tile, K-major.  Both forms make the same
// fp32 additions in the same order, so they give identical bits.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "gemm_relu_kernels.cuh"

namespace gemmrelu {
namespace splitk {

#ifndef GEMMRELU_SPLIT_KBS
#define GEMMRELU_SPLIT_KBS 4
#endif
// Stages of B (and A) each CTA asks L2 to fetch before it waits for the
// previous grid; 0 turns it off.
#ifndef GEMMRELU_SPLIT_PREFETCH
#define GEMMRELU_SPLIT_PREFETCH 4
#endif

constexpr int BNT = 128;     // N per tile (UMMA M, TMEM lanes)
constexpr int BK = 64;       // one 128-byte swizzle row of fp16
constexpr int UK = 16;       // K of one tcgen05.mma kind::f16
constexpr int kEpiWarps = 4;

// k blocks of 64 per pipeline stage for a given BMS: one stage moves B as two
// boxes of (64 * kbs) rows x 64 columns, so fewer and larger TMA copies carry
// the stream, while at least three stages fit in shared memory.  Work is
// split over K in whole stages ("super blocks").
__host__ __device__ constexpr int kbs_for(int bms) {
    return (GEMMRELU_SPLIT_KBS >= 4 && bms <= 32) ? 4
           : (GEMMRELU_SPLIT_KBS >= 2 && bms <= 64) ? 2
                                                   : 1;
}

// kCluster: a CTA pair (cluster of 2) computes all S pieces of a tile and
// adds them through distributed shared memory; the second CTA then needs a
// buffer of BMS x 128 fp32 for the first one's running sum.
template <int BMS, bool kCluster>
struct Cfg {
    static constexpr int kKbs = kbs_for(BMS);
    static constexpr int kSuperK = BK * kKbs;               // k per stage
    static constexpr uint32_t kBSlab = kSuperK * 64 * 2;    // (64 * kKbs) k-rows x 64 n
    static constexpr uint32_t kBTile = 2 * kBSlab;          // 128 n, N-major
    static constexpr uint32_t kASub = BMS * BK * 2;         // BMS rows x 64 k, K-major
    static constexpr uint32_t kATile = kKbs * kASub;
    static constexpr uint32_t kStageBytes = kBTile + kATile;
    static constexpr uint32_t kRedBytes = kCluster ? (uint32_t)BMS * BNT * 4u : 0u;
    static constexpr uint32_t kBudget = 227u * 1024u - 1024u - 256u - kRedBytes;
    static constexpr int kStagesRaw = (int)(kBudget / kStageBytes);
    static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
    static constexpr uint32_t kOffRed = kStages * kStageBytes;
    static constexpr uint32_t kOffBar = kOffRed + kRedBytes;
    static constexpr uint32_t kNumBars = 2 * kStages + 4 + 1 + 2;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
    // UMMA A (the B tile) N-major: bit 15 = 1; UMMA B (the A tile) K-major.
    static constexpr uint32_t kIdesc = make_idesc_f16_f32(BNT, BMS, 1, 0);
};

struct Params {
    float *part;                   // [S][M][N] fp32 partials (two-stage form)
    uint16_t *C;                   // output (cluster form)
    int M, N, K;
    int num_sb, splits;            // super blocks of kSuperK along K; S
    int64_t n_tiles, m_tiles, num_units;
    int split_major;               // unit order, see unit_coords
    int drop_arrive;
    uint64_t wait_limit_ns;
};

// One kernel, two forms.
//   kCluster = false: persistent CTAs walk work units (split s, n tile,
//     m tile) and write each unit's fp32 partial to part[s][m][n] (stage 1 of
//     the two-stage form).
//   kCluster = true (S even): the grid is made of CTA pairs (clusters of 2);
//     a pair walks tiles, CTA 0 computing pieces 0 .. S/2-1 of each and CTA 1
//     pieces S/2 .. S-1, every piece into its own TMEM accumulator.  CTA 0
//     adds its pieces in order, starting from 0, and writes that running sum
//     into CTA 1's shared memory (remote stores); CTA 1 continues the same
//     sum with its own pieces in order, applies the ReLU and stores fp16 C.
//     Every fp32 addition is the one the two-stage form's reduce kernel
//     makes, in the same order, so both forms give identical bits.
template <int BMS, bool kCluster>
__global__ void __launch_bounds__(192, 1)
    gemm_relu_splitk_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB, const Params p) {
    using G = Cfg<BMS, kCluster>;
    constexpr int kStages = G::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + G::kOffBar;
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (kStages + s); };
    auto accf_bar = [&](uint32_t b) { return bar0 + 8u * (2 * kStages + b); };
    auto acce_bar = [&](uint32_t b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    // cluster form: red_full (in CTA 1) completes when CTA 0 has written the
    // running sum of the current tile; red_empty (in CTA 0) when CTA 1 has
    // read the previous one.
    const uint32_t red_full = bar0 + 8u * (2 * kStages + 5);
    const uint32_t red_empty = bar0 + 8u * (2 * kStages + 6);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + G::kOffMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + G::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t S = p.splits;
    const uint32_t rank = kCluster ? cluster_ctarank() : 0u;
    // pieces per tile and CTA, each with its own accumulator (x2 buffers)
    const int pieces = kCluster ? (int)(S / 2) : 1;
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)(2 * pieces * BMS))
        tmem_cols <<= 1;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < (uint32_t)kStages; ++s) {
            mbar_init(full_bar(s), 1u);
            mbar_init(empty_bar(s), 1u);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1u);
            mbar_init(acce_bar(b), (uint32_t)kEpiWarps);
        }
        mbar_init(drain_bar, 1u);
        mbar_init(red_full, (uint32_t)kEpiWarps);
        mbar_init(red_empty, (uint32_t)kEpiWarps);
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();  // this thread's TMA copies may use them right away
        pdl_launch_dependents();
    }
    // Start-up.  The producer warp needs only its own barriers, so it signals
    // the other warps (named barrier 1) and, in the cluster form, the peer
    // CTA (cluster barrier), and starts loading at once; the MMA and epilogue
    // warps wait for the barrier initialisation, the TMEM allocation and --
    // before any remote access -- the peer's initialisation.
    uint32_t tmem_base = 0;
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_map(&tmA);
            tma_prefetch_map(&tmB);
        }
        __syncwarp();
        named_bar_arrive(1, 192);
        if constexpr (kCluster)
            cluster_arrive();
    } else {
        if (warp == 1) {
            tmem_alloc(smem_addr(tmem_slot), tmem_cols);
            tmem_relinquish();
        }
        tc_fence_before_sync();
        named_bar_sync(1, 192);
        tc_fence_after_sync();
        if constexpr (kCluster) {
            cluster_arrive();
            cluster_wait();
        }
        tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
        pdl_wait_primary();  // and the previous grid no longer reads C or the workspace
    }

    // Work unit u -> (first piece s, n tile, m tile) and its super blocks
    // [sb0, sb1).  Two-stage form: one piece per unit; split-major order has
    // neighbouring CTAs read neighbouring columns of the same rows of B,
    // split-minor order keeps the S pieces of one tile on neighbouring CTAs.
    // Cluster form: u is the tile, and the CTA's pieces are contiguous in k.
    const int64_t tiles = p.n_tiles * p.m_tiles;
    const int64_t u_first = kCluster ? (int64_t)(blockIdx.x / 2) : (int64_t)blockIdx.x;
    const int64_t u_stride = kCluster ? (int64_t)(gridDim.x / 2) : (int64_t)gridDim.x;
    auto piece_begin = [&](int64_t s) { return (int)((s * p.num_sb) / S); };
    auto unit_coords = [&](int64_t u, int64_t &s, int64_t &nt, int64_t &mt, int &sb0, int &sb1) {
        int64_t tile;
        if constexpr (kCluster) {
            s = (int64_t)rank * pieces;
            tile = u;
        } else {
            s = p.split_major ? u / tiles : u % S;
            tile = p.split_major ? u % tiles : u / S;
        }
        nt = tile % p.n_tiles;
        mt = tile / p.n_tiles;
        sb0 = piece_begin(s);
        sb1 = piece_begin(s + pieces);
    };

    if (warp == 0) {
        // ============================================================ TMA producer
        if (lane == 0) {
            // While the previous grid finishes, have L2 fetch the first
            // stages of this CTA's first unit: the launch-boundary gap in
            // the HBM stream then overlaps the previous grid's tail.
            if (GEMMRELU_SPLIT_PREFETCH > 0 && u_first < p.num_units) {
                int64_t s, nt, mt;
                int sb0, sb1;
                unit_coords(u_first, s, nt, mt, sb0, sb1);
                const int n0 = (int)(nt * BNT), m0 = (int)(mt * BMS);
                const int sb_end = min(sb1, sb0 + GEMMRELU_SPLIT_PREFETCH);
                for (int sb = sb0; sb < sb_end; ++sb) {
                    const int k0 = sb * G::kSuperK;
                    tma_prefetch_2d(&tmB, n0, k0);
                    tma_prefetch_2d(&tmB, n0 + 64, k0);
#pragma unroll
                    for (int i = 0; i < G::kKbs; ++i)
                        tma_prefetch_2d(&tmA, k0 + i * BK, m0);
                }
            }
            pdl_wait_primary();  // the previous grid's writes (A, B) are visible
            uint32_t stage = 0, phase = 0, parity = 0, issued = 0;
            bool ok = true;
            // B is read exactly once: stream it through L2 as evict-first
            const uint64_t stream_once = l2_policy_evict_first();
            for (int64_t u = u_first; ok && u < p.num_units; u += u_stride) {
                int64_t s, nt, mt;
                int sb0, sb1;
                unit_coords(u, s, nt, mt, sb0, sb1);
                const int n0 = (int)(nt * BNT), m0 = (int)(mt * BMS);
                for (int sb = sb0; sb < sb1; ++sb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_limit_ns, abort_flag,
                                      kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const bool drop =
                        p.drop_arrive && blockIdx.x == 0 && u == u_first && sb == sb0;
                    if (!drop) {
                        const uint32_t fb = full_bar(stage);
                        const uint32_t dst = base + stage * G::kStageBytes;
                        const int k0 = sb * G::kSuperK;
                        mbar_arrive_expect_tx(fb, G::kStageBytes);
                        tma_load_2d_hint(&tmB, dst, fb, n0, k0, stream_once);
                        tma_load_2d_hint(&tmB, dst + G::kBSlab, fb, n0 + 64, k0, stream_once);
#pragma unroll
                        for (int i = 0; i < G::kKbs; ++i)
                            tma_load_2d(&tmA, dst + G::kBTile + i * G::kASub, fb, k0 + i * BK, m0);
                        issued |= 1u << stage;
                        parity = (parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == (uint32_t)kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy issued must have landed before the CTA may exit
            for (uint32_t s = 0; s < (uint32_t)kStages; ++s)
                if (issued & (1u << s))
                    wait_drain(full_bar(s), (parity >> s) & 1u, p.wait_limit_ns, abort_flag);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int64_t i = 0;
            for (int64_t u = u_first; ok && u < p.num_units; u += u_stride, ++i) {
                int64_t s, nt, mt;
                int sb0, sb1;
                unit_coords(u, s, nt, mt, sb0, sb1);
                const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
                if (!wait_bounded(acce_bar(buf), use ^ 1u, p.wait_limit_ns, abort_flag,
                                  kSiteMmaAccEmpty))
                    break;
                tc_fence_after_sync();
                for (int j = 0; ok && j < pieces; ++j) {
                    // piece j of this unit: its own accumulator, started fresh
                    const int pb0 = piece_begin(s + j), pb1 = piece_begin(s + j + 1);
                    const uint32_t d = tmem_base + (buf * (uint32_t)pieces + (uint32_t)j) * BMS;
                    for (int sb = pb0; sb < pb1; ++sb) {
                        if (!wait_bounded(full_bar(stage), phase, p.wait_limit_ns, abort_flag,
                                          kSiteMmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t st = base + stage * G::kStageBytes;
#pragma unroll
                        for (int kk = 0; kk < G::kSuperK / UK; ++kk) {
                            // B slab rows are k: the next 16 k are 2 KB further;
                            // the two 64-wide N slabs are kBSlab apart (LBO).
                            const uint64_t adesc =
                                make_sdesc_sw128(st + kk * (UK * 128), G::kBSlab, 1024);
                            // A: 64-k sub-tile kk / 4, 32 bytes per 16 k inside it.
                            const uint64_t bdesc = make_sdesc_sw128(
                                st + G::kBTile + (kk / (BK / UK)) * G::kASub +
                                    (kk % (BK / UK)) * (UK * 2),
                                16, 1024);
                            umma_f16(d, adesc, bdesc, G::kIdesc,
                                     (sb > pb0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(empty_bar(stage));
                        if (++stage == (uint32_t)kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok)
                    break;
                umma_commit(accf_bar(buf));
            }
            // all MMAs of this thread complete before TMEM can be released
            umma_commit(drain_bar);
            wait_drain(drain_bar, 0u, p.wait_limit_ns, abort_flag);
        }
    } else {
        // ============================================================ epilogue
        // Lane l of warp q holds output column n = n0 + 32q + l (a TMEM lane)
        // and BMS rows m0.. (TMEM columns); for each row the warp stores 32
        // consecutive floats (128 B): to part[s][m][*] (two-stage form), or
        // the pair's running sum to CTA 1's buffer (cluster form, CTA 0).
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        int64_t i = 0;
        for (int64_t u = u_first; u < p.num_units; u += u_stride, ++i) {
            int64_t s, nt, mt;
            int sb0, sb1;
            unit_coords(u, s, nt, mt, sb0, sb1);
            const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
            const bool ok = wait_bounded(accf_bar(buf), use, p.wait_limit_ns, abort_flag,
                                         kSiteEpiAccFull);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after_sync();
            if constexpr (kCluster) {
                // CTA 1's buffer: the running sum over CTA 0's pieces,
                // [m][n] fp32 (row m of the tile, column n = TMEM lane).
                const uint32_t red = base + G::kOffRed;
                const uint32_t n_local = (uint32_t)(32 * q + lane);
                const uint32_t acc0 = tmem_base + lane_base + buf * (uint32_t)pieces * BMS;
                if (rank == 0) {
                    // CTA 1 has read the previous tile's sum
                    const bool freed = wait_bounded_cluster(red_empty, (uint32_t)((i & 1) ^ 1),
                                                            p.wait_limit_ns, abort_flag,
                                                            kSiteClusterReduce);
                    if (!__all_sync(0xffffffffu, freed))
                        break;
                    const uint32_t peer_red = mapa_shared(red, 1u);
#pragma unroll 1
                    for (int c0 = 0; c0 < BMS; c0 += 16) {
                        float acc[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            acc[c] = 0.0f;
#pragma unroll 1
                        for (int j = 0; j < pieces; ++j) {
                            uint32_t r[16];
                            tmem_ld_x16_sync(acc0 + (uint32_t)j * BMS + c0, r);
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                acc[c] += __uint_as_float(r[c]);
                        }
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            st_cluster_f32(peer_red + 4u * ((uint32_t)(c0 + c) * BNT + n_local),
                                           acc[c]);
                    }
                    // accumulators read: hand them back to the MMA warp
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(acce_bar(buf));
                    // publish: each lane orders its remote stores, the warp
                    // synchronises, lane 0 signals CTA 1 (release, cluster scope)
                    fence_acq_rel_cluster();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_cluster(mapa_shared(red_full, 1u));
                } else {
                    const bool full = wait_bounded_cluster(red_full, (uint32_t)(i & 1),
                                                           p.wait_limit_ns, abort_flag,
                                                           kSiteClusterReduce);
                    if (!__all_sync(0xffffffffu, full))
                        break;
                    const int64_t col = nt * BNT + n_local;
#pragma unroll 1
                    for (int c0 = 0; c0 < BMS; c0 += 16) {
                        float acc[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            acc[c] = __uint_as_float(
                                ld_shared_b32(red + 4u * ((uint32_t)(c0 + c) * BNT + n_local)));
#pragma unroll 1
                        for (int j = 0; j < pieces; ++j) {
                            uint32_t r[16];
                            tmem_ld_x16_sync(acc0 + (uint32_t)j * BMS + c0, r);
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                acc[c] += __uint_as_float(r[c]);
                        }
                        if (col < p.N) {
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const int64_t m = mt * BMS + c0 + c;
                                if (m < p.M)
                                    p.C[m * p.N + col] = (uint16_t)(
                                        relu_pack_half2(__float_as_uint(acc[c]), 0u) & 0xffffu);
                            }
                        }
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(acce_bar(buf));
                    // buffer read: CTA 0 may write the next tile's sum
                    fence_acq_rel_cluster();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_cluster(mapa_shared(red_empty, 0u));
                }
                continue;
            }
            const int64_t n = nt * BNT + 32 * q + lane;
            const int64_t m0 = mt * BMS;
            float *part = p.part + (size_t)s * p.M * p.N;
#pragma unroll 1
            for (int c0 = 0; c0 < BMS; c0 += 16) {
                uint32_t r[16];
                tmem_ld_x16_sync(tmem_base + lane_base + buf * BMS + c0, r);
                if (n < p.N) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int64_t m = m0 + c0 + c;
                        if (m < p.M)
                            part[m * p.N + n] = __uint_as_float(r[c]);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acce_bar(buf));
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kCluster) {
        if (warp == 0)
            cluster_wait();  // the start-up phase the producer only arrived on
        cluster_sync();      // no CTA leaves while the other may still access its shared memory
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

// Stage 2: C[m][n] = fp16(max(part[0][m][n] + part[1][m][n] + ... +
// part[S-1][m][n], 0)), accumulated in fp32 in exactly that order.  Each
// thread handles four consecutive n (N is a multiple of 8 on this path): the
// loads of up to eight splits (one float4 each) are all issued before the
// first add, so a thread waits for about one memory round trip per eight
// splits; the store is one 8-byte vector when C is 8-byte aligned.
__global__ void __launch_bounds__(256)
    gemm_relu_splitk_reduce_kernel(const float *__restrict__ part, uint16_t *__restrict__ C, int M,
                                   int N, int S, int c_vec8) {
    if (threadIdx.x == 0)
        pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t per_row = N / 4;
    const int64_t groups = (int64_t)M * per_row;
    const size_t split_stride = (size_t)M * (size_t)N;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = g / per_row;
        const int64_t n = (g - m * per_row) * 4;
        const float *src = part + m * N + n;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int s0 = 0; s0 < S; s0 += 8) {
            float4 v[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                v[t] = (s0 + t < S) ? __ldcg(reinterpret_cast<const float4 *>(
                                          src + (size_t)(s0 + t) * split_stride))
                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (s0 + t < S) {
                    acc.x += v[t].x;
                    acc.y += v[t].y;
                    acc.z += v[t].z;
                    acc.w += v[t].w;
                }
            }
        }
        const uint32_t h0 = relu_pack_half2(__float_as_uint(acc.x), __float_as_uint(acc.y));
        const uint32_t h1 = relu_pack_half2(__float_as_uint(acc.z), __float_as_uint(acc.w));
        uint16_t *dst = C + m * N + n;
        if (c_vec8) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(h0, h1);
        } else {
            dst[0] = (uint16_t)(h0 & 0xffffu);
            dst[1] = (uint16_t)(h0 >> 16);
            dst[2] = (uint16_t)(h1 & 0xffffu);
            dst[3] = (uint16_t)(h1 >> 16);
        }
    }
}

}  // namespace splitk
}  // namespace gemmrelu
