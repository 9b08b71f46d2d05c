// flash_attention.cuh -- attention forward, O = softmax(Q K^T / sqrt(d)) V,
// for fp16 Q, K, V, O in the [batch][seq][heads][dim] layout, fp32 inside.
//
// The FlashAttention section of the TileLang tutorial pages: never form the
// seq x seq scores; stream K/V blocks and keep, per query row, a running
// maximum m, a running denominator l and an unnormalised output, rescaling
// the output by 2^(m_old - m_new) when the maximum moves; exponentials in
// base 2 with alpha = log2(e) / sqrt(d) folded into the scores; only P, the
// matrix fed to the second product, is rounded to fp16; causal mode stops at
// the diagonal block and masks its strictly upper triangle.
//
// On sm_103a one CTA owns two 128-row query tiles (t = 0, 1) of one
// (batch, head) and ping-pongs them so that the tensor core works on one
// tile while the other's softmax runs:
//   warps 0-3   softmax of tile 0, one thread per query row (its TMEM lane);
//   warps 4-7   softmax of tile 1;
//   warp 8      TMA: both Q tiles once, then K and V blocks of 128 keys into
//               a 2-stage ring (4-D tensor maps over the bshd layout, 64-wide
//               128-byte-swizzled boxes);
//   warp 9      one thread issues tcgen05.mma in the order
//                 S0_0, S1_0, { PV0_j, S0_j+1, PV1_j, S1_j+1 } for j = 0, 1, ...
//               with S_t = Q_t K_j^T in TMEM and O_t += P_t V_j, P_t read
//               from TMEM (the softmax writes it over the scores it has read).
// TMEM columns: S0 / P0 at 0, S1 / P1 at 128, O0 at 256, O1 at 256 + d.
// A score MMA for tile t is issued only after the P V MMA that reads P_t,
// and tcgen05 operations of one thread execute in issue order.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "gemm_relu_kernels.cuh"

namespace gemmrelu {
namespace attn {

constexpr int BM = 128;          // query rows per tile (UMMA M, TMEM lanes)
constexpr int BN = 128;          // keys per block
constexpr int UKA = 16;          // K of one tcgen05.mma kind::f16
constexpr int kKV = 2;           // K/V ring stages
constexpr int kTiles = 2;        // query tiles per CTA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kSub = BM * 128;   // one [128 rows][64] fp16 swizzled sub-tile: 16 KB

template <int HD>
struct Cfg {
    static_assert(HD == 64 || HD == 128, "head dim 64 or 128");
    static constexpr int kDSub = HD / 64;
    static constexpr uint32_t kQBytes = kDSub * kSub;   // [128 q][HD]: K-major sub-tiles
    static constexpr uint32_t kKBytes = kDSub * kSub;   // [128 keys][HD]: K-major sub-tiles
    static constexpr uint32_t kVBytes = kDSub * kSub;   // [128 keys][HD]: N-major 64-wide slabs
    static constexpr uint32_t kOffQ = 0;                // + t * kQBytes
    static constexpr uint32_t kOffK = kOffQ + kTiles * kQBytes;
    static constexpr uint32_t kOffV = kOffK + kKV * kKBytes;
    static constexpr uint32_t kOffBar = kOffV + kKV * kVBytes;
    // q_full, k_full[kKV], v_full[kKV], kv_empty[kKV], s_full[2], p_full[2],
    // o_full, drain
    static constexpr uint32_t kNumBars = 1 + 3 * kKV + 2 + 2 + 2;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmemS = 0;               // + t * BN
    static constexpr uint32_t kTmemO = 2 * BN;          // + t * HD
    // S = Q K^T: both K-major.  O += P V: P from TMEM (K-major), V N-major.
    static constexpr uint32_t kIdescS = make_idesc_f16_f32(BM, BN, 0, 0);
    static constexpr uint32_t kIdescO = make_idesc_f16_f32(BM, HD, 0, 1);
};

struct Params {
    uint16_t *O;           // [batch][seq][heads][dim] fp16
    int batch, seq, heads;
    int q_tiles;           // ceil(seq / BM)
    int ctas_x;            // ceil(q_tiles / 2)
    int causal;
    float scale;           // log2(e) / sqrt(dim)
    int drop_arrive;
    uint64_t wait_limit_ns;
};

// 2^x by the hardware's base-2 exponential (approximate, relative error near
// 2^-22; flushes subnormal results to zero) -- ample for P, which is then
// rounded to fp16.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The running maximum used as the exponent reference moves (and the output
// is rescaled) only when a row's maximum exceeds it by more than this many
// units of log2: P then stays below 2^8, well inside fp16, and the
// normalisation by the same reference keeps the result exact up to rounding.
constexpr float kRescaleLog2 = 8.0f;

// Pack two fp32 values as an fp16 pair (round to nearest even), low = a.
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    flash_attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                               const __grid_constant__ CUtensorMap tmK,
                               const __grid_constant__ CUtensorMap tmV, const Params p) {
    using G = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t bar0 = base + G::kOffBar;
    const uint32_t q_full = bar0;
    auto k_full = [&](uint32_t s) { return bar0 + 8u * (1 + s); };
    auto v_full = [&](uint32_t s) { return bar0 + 8u * (1 + kKV + s); };
    auto kv_empty = [&](uint32_t s) { return bar0 + 8u * (1 + 2 * kKV + s); };
    auto s_full = [&](uint32_t t) { return bar0 + 8u * (1 + 3 * kKV + t); };
    auto p_full = [&](uint32_t t) { return bar0 + 8u * (3 + 3 * kKV + t); };
    const uint32_t o_full = bar0 + 8u * (5 + 3 * kKV);
    const uint32_t drain_bar = bar0 + 8u * (6 + 3 * kKV);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + G::kOffMisc);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + G::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // heaviest tile pairs first in causal mode
    const int pair = p.causal ? (p.ctas_x - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const int head = blockIdx.y, batch = blockIdx.z;
    const int kv_all = (p.seq + BN - 1) / BN;
    // tiles 2 * pair and 2 * pair + 1; their numbers of key blocks
    const int tile0 = kTiles * pair, tile1 = tile0 + 1;
    auto blocks_of = [&](int tl) { return p.causal ? (tl + 1 < kv_all ? tl + 1 : kv_all) : kv_all; };
    const int nb0 = blocks_of(tile0);
    const int nb1 = tile1 < p.q_tiles ? blocks_of(tile1) : nb0;  // a padding tile: rows not stored
    const int nb = nb1 > nb0 ? nb1 : nb0;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1u);
        for (uint32_t s = 0; s < (uint32_t)kKV; ++s) {
            mbar_init(k_full(s), 1u);
            mbar_init(v_full(s), 1u);
            mbar_init(kv_empty(s), 1u);
        }
        for (uint32_t t = 0; t < (uint32_t)kTiles; ++t) {
            mbar_init(s_full(t), 1u);
            mbar_init(p_full(t), 4u);
        }
        mbar_init(o_full, 1u);
        mbar_init(drain_bar, 1u);
        *abort_flag = 0u;
        fence_mbar_init();
        pdl_launch_dependents();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), G::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    pdl_wait_primary();  // the previous grid of the stream has completed

    if (warp == kProducerWarp) {
        // ============================================================ TMA producer
        if (lane == 0) {
            uint32_t issued = 0, parity = 0;  // K/V stages with copies in flight
            bool q_issued = false;
            if (!(p.drop_arrive && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)) {
                mbar_arrive_expect_tx(q_full, kTiles * G::kQBytes);
                for (int t = 0; t < kTiles; ++t)
#pragma unroll
                    for (int d = 0; d < G::kDSub; ++d)
                        tma_load_4d(&tmQ, base + G::kOffQ + t * G::kQBytes + d * kSub, q_full,
                                    64 * d, head, (tile0 + t) * BM, batch);
                q_issued = true;
            }
            for (int j = 0; j < nb; ++j) {
                const uint32_t st = (uint32_t)(j % kKV), ph = (uint32_t)((j / kKV) & 1);
                if (!wait_bounded_eager(kv_empty(st), ph ^ 1u, p.wait_limit_ns, abort_flag,
                                  kSiteProducerEmpty))
                    break;
                mbar_arrive_expect_tx(k_full(st), G::kKBytes);
#pragma unroll
                for (int d = 0; d < G::kDSub; ++d)
                    tma_load_4d(&tmK, base + G::kOffK + st * G::kKBytes + d * kSub, k_full(st),
                                64 * d, head, j * BN, batch);
                mbar_arrive_expect_tx(v_full(st), G::kVBytes);
#pragma unroll
                for (int d = 0; d < G::kDSub; ++d)
                    tma_load_4d(&tmV, base + G::kOffV + st * G::kVBytes + d * kSub, v_full(st),
                                64 * d, head, j * BN, batch);
                issued |= 1u << st;
                parity = (parity & ~(1u << st)) | (ph << st);
            }
            // every copy issued must have landed before the CTA may exit
            if (q_issued)
                wait_drain(q_full, 0u, p.wait_limit_ns, abort_flag);
            for (uint32_t s = 0; s < (uint32_t)kKV; ++s)
                if (issued & (1u << s)) {
                    wait_drain(k_full(s), (parity >> s) & 1u, p.wait_limit_ns, abort_flag);
                    wait_drain(v_full(s), (parity >> s) & 1u, p.wait_limit_ns, abort_flag);
                }
        }
    } else if (warp == kMmaWarp) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            bool ok = wait_bounded_eager(q_full, 0u, p.wait_limit_ns, abort_flag, kSiteMmaFull);
            // S_t = Q_t K_j^T
            auto score = [&](int t, int j) -> bool {
                const uint32_t st = (uint32_t)(j % kKV), ph = (uint32_t)((j / kKV) & 1);
                if (!wait_bounded_eager(k_full(st), ph, p.wait_limit_ns, abort_flag, kSiteMmaFull))
                    return false;
                tc_fence_after_sync();
                // descriptors built once, advanced in their 16-byte units:
                // 32 bytes per 16 k inside a 64-wide sub-tile, kSub across
                const uint64_t qd = make_sdesc_sw128(base + G::kOffQ + t * G::kQBytes, 16, 1024);
                const uint64_t kd = make_sdesc_sw128(base + G::kOffK + st * G::kKBytes, 16, 1024);
                const uint32_t d_s = tmem_base + G::kTmemS + t * BN;
#pragma unroll
                for (int kk = 0; kk < HD / UKA; ++kk) {
                    const uint64_t off = (uint64_t)((kk / 4) * (kSub >> 4) + (kk % 4) * 2);
                    umma_f16(d_s, qd + off, kd + off, G::kIdescS, kk > 0 ? 1u : 0u);
                }
                umma_commit(s_full(t));
                return true;
            };
            // O_t += P_t V_j, P_t from TMEM (over S_t)
            auto pv = [&](int t, int j) -> bool {
                const uint32_t st = (uint32_t)(j % kKV), ph = (uint32_t)((j / kKV) & 1);
                if (!wait_bounded_eager(p_full(t), (uint32_t)(j & 1), p.wait_limit_ns, abort_flag,
                                  kSiteMmaAccEmpty) ||
                    !wait_bounded_eager(v_full(st), ph, p.wait_limit_ns, abort_flag, kSiteMmaFull))
                    return false;
                tc_fence_after_sync();
                // V descriptor advanced 16 key rows (2 KB) per step; P columns 8
                const uint64_t vd = make_sdesc_sw128(base + G::kOffV + st * G::kVBytes, kSub, 1024);
                const uint32_t d_o = tmem_base + G::kTmemO + t * HD;
                const uint32_t a_p = tmem_base + G::kTmemS + t * BN;
#pragma unroll
                for (int kk = 0; kk < BN / UKA; ++kk)
                    umma_f16_ts(d_o, a_p + kk * (UKA / 2), vd + (uint64_t)(kk * ((UKA * 128) >> 4)),
                                G::kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                return true;
            };
            if (ok)
                ok = score(0, 0) && score(1, 0);
            for (int j = 0; ok && j < nb; ++j) {
                if (j < nb0) {
                    ok = pv(0, j) && (j + 1 >= nb0 || score(0, j + 1));
                    if (!ok)
                        break;
                }
                ok = pv(1, j);
                if (!ok)
                    break;
                umma_commit(kv_empty((uint32_t)(j % kKV)));
                if (j + 1 < nb1)
                    ok = score(1, j + 1);
            }
            if (ok)
                umma_commit(o_full);
            // all MMAs of this thread complete before TMEM can be released
            umma_commit(drain_bar);
            wait_drain(drain_bar, 0u, p.wait_limit_ns, abort_flag);
        }
    } else {
        // ============================================================ softmax / output
        const int t = warp >> 2;                        // query tile
        const int q = warp & 3;                         // TMEM lanes 32q .. 32q+31
        const int r = 32 * q + lane;                    // query row in the tile
        const int qi = (tile0 + t) * BM + r;            // query index in the sequence
        const int my_nb = t == 0 ? nb0 : nb1;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t s_addr = tmem_base + lane_base + G::kTmemS + t * BN;
        const uint32_t o_addr = tmem_base + lane_base + G::kTmemO + t * HD;
        const int kmax = p.causal ? (qi + 1 < p.seq ? qi + 1 : p.seq) : p.seq;
        float m = -INFINITY, l = 0.0f;
        bool alive = true;
        for (int j = 0; j < my_nb; ++j) {
            const bool ok = wait_bounded_eager(s_full((uint32_t)t), (uint32_t)(j & 1), p.wait_limit_ns,
                                         abort_flag, kSiteEpiAccFull);
            if (!__all_sync(0xffffffffu, ok)) {
                alive = false;
                break;
            }
            tc_fence_after_sync();
            // keys past the sequence, and (causal) keys after the query
            const bool masked = (j + 1) * BN > p.seq || (p.causal && j == my_nb - 1);
            const int key0 = j * BN;
            // the row's 128 scores: one TMEM round trip, kept in registers
            uint32_t v[BN];
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32)
                tmem_ld_x32(s_addr + c0, *reinterpret_cast<uint32_t(*)[32]>(&v[c0]));
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32)
                tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&v[c0]));
            if (masked) {
#pragma unroll
                for (int i = 0; i < BN; ++i)
                    v[i] = key0 + i < kmax ? v[i] : __float_as_uint(-INFINITY);
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int i = 0; i < BN; i += 2) {
                mx0 = fmaxf(mx0, __uint_as_float(v[i]));
                mx1 = fmaxf(mx1, __uint_as_float(v[i + 1]));
            }
            const float m_blk = fmaxf(mx0, mx1) * p.scale;   // scale > 0
            // move the reference only when the maximum grew by more than
            // kRescaleLog2 (always at the first block)
            const bool move = m_blk > m + kRescaleLog2;
            const float m_ref = move ? m_blk : m;
            const float alpha = move ? fast_exp2(m - m_ref) : 1.0f;   // 0 at the first block
            // exponentials (masked scores are -inf: 2^-inf = 0), their sum,
            // and P as fp16 over the scores
            // (pairs of fp32 lanes per instruction: __ffma2_rn / __fadd2_rn
            // round each lane as fmaf / + would)
            const float2 sc2 = make_float2(p.scale, p.scale), nm2 = make_float2(-m_ref, -m_ref);
            float2 sa = make_float2(0.0f, 0.0f), sb = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t ph[16];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float2 x01 = __ffma2_rn(
                        make_float2(__uint_as_float(v[c0 + i]), __uint_as_float(v[c0 + i + 1])), sc2, nm2);
                    const float2 x23 = __ffma2_rn(
                        make_float2(__uint_as_float(v[c0 + i + 2]), __uint_as_float(v[c0 + i + 3])), sc2, nm2);
                    const float2 e01 = make_float2(fast_exp2(x01.x), fast_exp2(x01.y));
                    const float2 e23 = make_float2(fast_exp2(x23.x), fast_exp2(x23.y));
                    sa = __fadd2_rn(sa, e01);
                    sb = __fadd2_rn(sb, e23);
                    ph[i / 2] = pack_half2(e01.x, e01.y);
                    ph[i / 2 + 1] = pack_half2(e23.x, e23.y);
                }
                tmem_st_x16(s_addr + c0 / 2, ph);
            }
            l = l * alpha + ((sa.x + sa.y) + (sb.x + sb.y));
            m = m_ref;
            // rescale this warp's output rows when any of their references moved
            // (the previous P V of this tile completed before S_j was written)
            if (j >= 1 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_x32_sync(o_addr + c0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st_x32(o_addr + c0, v);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(p_full((uint32_t)t));
        }
        // the last P V of both tiles, then O / l rounded to fp16
        if (alive) {
            const bool done = wait_bounded_eager(o_full, 0u, p.wait_limit_ns, abort_flag,
                                           kSiteEpiAccFull);
            if (__all_sync(0xffffffffu, done)) {
                tc_fence_after_sync();
                const float inv_l = 1.0f / l;
                uint16_t *dst = p.O + (((int64_t)batch * p.seq + qi) * p.heads + head) * HD;
#pragma unroll 1
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_x32_sync(o_addr + c0, v);
                    uint32_t h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        h[i] = pack_half2(__uint_as_float(v[2 * i]) * inv_l,
                                          __uint_as_float(v[2 * i + 1]) * inv_l);
                    if (qi < p.seq) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, G::kTmemCols);
    }
}

}  // namespace attn
}  // namespace gemmrelu
