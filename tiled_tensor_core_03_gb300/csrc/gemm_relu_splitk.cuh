// gemm_relu_splitk.cuh -- split-K fused GEMM + ReLU for skinny (memory-bound)
// shapes, in two stages.
//
// The split-K scheme of "TileLang 编程基本知识点" section 5.1 cuts the K range
// into S pieces computed by different CTAs; each piece only offsets K.  The
// page adds the fp32 partials with atomics into a pre-zeroed C, and notes
// that for reproducible results the partials should instead be written to a
// workspace and reduced in a separate step.  That is what happens here:
//
//   stage 1  gemm_relu_splitk_partial_kernel: C^T = B^T . A^T per piece.  The
//            MMA's M side (128 TMEM lanes) runs over N and its narrow N side
//            (BMS columns) over M, so M = 16 costs a 128 x 16 MMA instead of
//            a mostly empty 128-row tile.  UMMA A operand = a B tile,
//            N-major; UMMA B operand = an A tile, K-major.  Each work unit
//            (split s, n tile, m tile) writes its raw fp32 partial (no ReLU)
//            to part[s][m][n].
//   stage 2  gemm_relu_splitk_reduce_kernel: C[m][n] = fp16(max(sum over
//            s = 0..S-1 of part[s][m][n], 0)), summed in that fixed order, so
//            the result is bit-identical from run to run.
//
// Stage 2 is launched as a programmatic dependent of stage 1: its CTAs
// become resident as stage-1 CTAs retire and wait (griddepcontrol.wait)
// until stage 1 has completed and its writes are visible.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "gemm_relu_kernels.cuh"

namespace gemmrelu {
namespace splitk {

#ifndef GEMMRELU_SPLIT_KBS
#define GEMMRELU_SPLIT_KBS 4
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

template <int BMS>
struct Cfg {
    static constexpr int kKbs = kbs_for(BMS);
    static constexpr int kSuperK = BK * kKbs;               // k per stage
    static constexpr uint32_t kBSlab = kSuperK * 64 * 2;    // (64 * kKbs) k-rows x 64 n
    static constexpr uint32_t kBTile = 2 * kBSlab;          // 128 n, N-major
    static constexpr uint32_t kASub = BMS * BK * 2;         // BMS rows x 64 k, K-major
    static constexpr uint32_t kATile = kKbs * kASub;
    static constexpr uint32_t kStageBytes = kBTile + kATile;
    static constexpr uint32_t kBudget = 227u * 1024u - 1024u - 256u;
    static constexpr int kStagesRaw = (int)(kBudget / kStageBytes);
    static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
    static constexpr uint32_t kOffBar = kStages * kStageBytes;
    static constexpr uint32_t kNumBars = 2 * kStages + 4 + 1;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
    static constexpr uint32_t kTmemCols = (2 * BMS < 32) ? 32 : 2 * BMS;  // power of 2
    // UMMA A (the B tile) N-major: bit 15 = 1; UMMA B (the A tile) K-major.
    static constexpr uint32_t kIdesc = make_idesc_f16_f32(BNT, BMS, 1, 0);
};

struct Params {
    float *part;                   // [S][M][N] fp32 partials
    int M, N, K;
    int num_sb, splits;            // super blocks of kSuperK along K; S
    int64_t n_tiles, m_tiles, num_units;
    int split_major;               // unit order, see unit_coords
    int drop_arrive;
    uint64_t wait_limit_ns;
};

// Let the dependent (reduce) grid launch early; it waits for this grid's
// completion itself.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the grid this one depends on has completed and its memory
// operations are visible (returns at once without such a dependency).
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int BMS>
__global__ void __launch_bounds__(192, 1)
    gemm_relu_splitk_partial_kernel(const __grid_constant__ CUtensorMap tmA,
                                    const __grid_constant__ CUtensorMap tmB, const Params p) {
    using G = Cfg<BMS>;
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
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + G::kOffMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + G::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t S = p.splits;

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
        *abort_flag = 0u;
        fence_mbar_init();
        pdl_launch_dependents();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), G::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

    // Work unit u -> (split s, n tile, m tile).  Split-major order has
    // neighbouring CTAs read neighbouring columns of the same rows of B;
    // split-minor order keeps the S pieces of one tile on neighbouring CTAs.
    const int64_t tiles = p.n_tiles * p.m_tiles;
    auto unit_coords = [&](int64_t u, int64_t &s, int64_t &nt, int64_t &mt, int &sb0, int &sb1) {
        s = p.split_major ? u / tiles : u % S;
        const int64_t tile = p.split_major ? u % tiles : u / S;
        nt = tile % p.n_tiles;
        mt = tile / p.n_tiles;
        sb0 = (int)((s * p.num_sb) / S);
        sb1 = (int)(((s + 1) * p.num_sb) / S);
    };

    if (warp == 0) {
        // ============================================================ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, parity = 0, issued = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
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
                        p.drop_arrive && blockIdx.x == 0 && u == blockIdx.x && sb == sb0;
                    if (!drop) {
                        const uint32_t fb = full_bar(stage);
                        const uint32_t dst = base + stage * G::kStageBytes;
                        const int k0 = sb * G::kSuperK;
                        mbar_arrive_expect_tx(fb, G::kStageBytes);
                        tma_load_2d(&tmB, dst, fb, n0, k0);
                        tma_load_2d(&tmB, dst + G::kBSlab, fb, n0 + 64, k0);
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
            for (int64_t u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++i) {
                int64_t s, nt, mt;
                int sb0, sb1;
                unit_coords(u, s, nt, mt, sb0, sb1);
                const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
                if (!wait_bounded(acce_bar(buf), use ^ 1u, p.wait_limit_ns, abort_flag,
                                  kSiteMmaAccEmpty))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + buf * BMS;
                for (int sb = sb0; sb < sb1; ++sb) {
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
                            st + G::kBTile + (kk / (BK / UK)) * G::kASub + (kk % (BK / UK)) * (UK * 2),
                            16, 1024);
                        umma_f16(d, adesc, bdesc, G::kIdesc, (sb > sb0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(empty_bar(stage));
                    if (++stage == (uint32_t)kStages) {
                        stage = 0;
                        phase ^= 1u;
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
        // consecutive floats (128 B) of part[s][m][*].
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        int64_t i = 0;
        for (int64_t u = blockIdx.x; u < p.num_units; u += gridDim.x, ++i) {
            int64_t s, nt, mt;
            int sb0, sb1;
            unit_coords(u, s, nt, mt, sb0, sb1);
            const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
            const bool ok = wait_bounded(accf_bar(buf), use, p.wait_limit_ns, abort_flag,
                                         kSiteEpiAccFull);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after_sync();
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
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, G::kTmemCols);
    }
}

// Stage 2: C[m][n] = fp16(max(part[0][m][n] + part[1][m][n] + ... +
// part[S-1][m][n], 0)), accumulated in fp32 in exactly that order.  Each
// thread handles eight consecutive n (N is a multiple of 8 on this path), so
// loads are 32-byte float4 pairs and the store is one 16-byte vector when C
// is 16-byte aligned.  Loads of four splits are issued before they are added.
__global__ void __launch_bounds__(256)
    gemm_relu_splitk_reduce_kernel(const float *__restrict__ part, uint16_t *__restrict__ C, int M,
                                   int N, int S, int c_vec16) {
    pdl_wait_primary();
    const int64_t per_row = N / 8;
    const int64_t groups = (int64_t)M * per_row;
    const size_t split_stride = (size_t)M * (size_t)N;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = g / per_row;
        const int64_t n = (g - m * per_row) * 8;
        const float *src = part + m * N + n;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[j] = 0.0f;
        int s = 0;
        for (; s + 4 <= S; s += 4) {
            float4 v[4][2];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float4 *q = reinterpret_cast<const float4 *>(src + (size_t)(s + t) * split_stride);
                v[t][0] = __ldcg(q);
                v[t][1] = __ldcg(q + 1);
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                acc[0] += v[t][0].x; acc[1] += v[t][0].y; acc[2] += v[t][0].z; acc[3] += v[t][0].w;
                acc[4] += v[t][1].x; acc[5] += v[t][1].y; acc[6] += v[t][1].z; acc[7] += v[t][1].w;
            }
        }
        for (; s < S; ++s) {
            const float4 *q = reinterpret_cast<const float4 *>(src + (size_t)s * split_stride);
            const float4 a = __ldcg(q), b = __ldcg(q + 1);
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            h[j] = relu_pack_half2(__float_as_uint(acc[2 * j]), __float_as_uint(acc[2 * j + 1]));
        uint16_t *dst = C + m * N + n;
        if (c_vec16) {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                dst[2 * j] = (uint16_t)(h[j] & 0xffffu);
                dst[2 * j + 1] = (uint16_t)(h[j] >> 16);
            }
        }
    }
}

}  // namespace splitk
}  // namespace gemmrelu
