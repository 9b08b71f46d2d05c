// gemm_relu_2sm.cuh -- the fused fp16 GEMM + ReLU on CTA pairs (2-SM MMA).
//
// Same operation and epilogue as the fused kernel of gemm_relu_kernels.cuh:
// C = fp16(max(A . B, 0)), fp32 accumulation, ReLU on the accumulator.  What
// changes is the tile: a cluster of two CTAs (on the two SMs of a TPC)
// computes one 256 x 256 output tile with tcgen05.mma.cta_group::2.
//
//   CTA rank r of the pair loads A rows [m0 + 128 r, +128) and B columns
//   [n0 + 128 r, +128) of every 64-wide k block into its own shared memory;
//   one thread of the even CTA issues the 256 x 256 x 16 MMAs, which read
//   A rows and B columns from both CTAs and leave rows [128 r, +128) of the
//   fp32 accumulator in CTA r's TMEM.  Each CTA's epilogue stores its own
//   128 rows.
//
// Why: with one CTA per 128 x 256 tile, every k block costs 48 KB of TMA
// writes plus 48 KB of MMA reads of shared memory, more than the 512 MMA
// cycles can absorb at 128 B/clk, so the tensor pipe idled about a third of
// the time (measured on GB300).  Here each SM holds 32 KB per k block for the
// same MMA work per SM, which the shared-memory port can sustain.
//
// Pair protocol: the even CTA owns the pipeline barriers that gate its MMA.
// Both CTAs' TMA loads complete on the even CTA's full[stage] barrier (which
// expects the bytes of both); the MMA commit arrives on empty[stage] and
// acc_full[buf] in both CTAs (multicast); both CTAs' epilogue warps arrive on
// the even CTA's acc_empty[buf] (8 arrivals).  Every wait stays bounded as in
// the single-CTA kernel; both CTAs always meet at the final cluster barrier.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "gemm_relu_kernels.cuh"

namespace gemmrelu {
namespace pair {

using fused::BK;
using fused::UK;
using fused::kATile;      // 128 rows x 64 k of A per CTA (16 KB)
using fused::kBSlab;      // 64 k x 64 n of B (8 KB)
using fused::kEpiBuf;
using fused::kEpiWarps;
using fused::SkShape;
using fused::sk_num_items;
using fused::sk_item_at;
using fused::kItemFull;
using fused::kItemPieceIn;
using fused::kItemPieceOut;

constexpr int BMP = 256;                        // tile rows (both CTAs)
constexpr int BNP = 256;                        // tile columns (UMMA N)
constexpr int kBHalf = 128;                     // B columns held per CTA
constexpr uint32_t kBTile = BK * kBHalf * 2;    // 16 KB = 2 slabs per CTA
constexpr uint32_t kStageBytes = kATile + kBTile;   // 32 KB per CTA
constexpr int kStages = 6;
constexpr uint32_t kTmemCols = 2 * BNP;         // double-buffered 128 x 256 fp32

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kATile;
constexpr uint32_t kOffEpi = kOffB + kStages * kBTile;
constexpr uint32_t kOffBar = kOffEpi + kEpiWarps * 2 * kEpiBuf;
constexpr uint32_t kNumBars = 2 * kStages + 4 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 227u * 1024u, "pair kernel: shared memory over the per-CTA limit");

// A K-major, B N-major; M = 256 across the pair, N = 256.
constexpr uint32_t kIdesc = make_idesc_f16_f32(BMP, BNP, 0, 1);
constexpr int kThreads = 192;                   // producer, MMA, 4 epilogue warps

struct Params {
    uint16_t *C;                                // for predicated stores (kTmaStore false)
    int M, N, K;
    int num_kb;
    int64_t m_tiles, n_tiles, num_tiles;        // 256 x 256 tiles
    int panel;
    int drop_arrive;
    uint64_t wait_limit_ns;
    // Stream-K over pairs, as in the single-CTA kernel: tiles [0, dp_tiles)
    // data-parallel, the k blocks of the rest cut into one range per pair.
    // CTA b and CTA b + 2 (the same half of the next pair) meet on the rows
    // of a cut tile through the wait-free exchange of the single-CTA kernel
    // (fused::sk_exchange): k tail in sk_part[b + 2], k head in sk_head[b],
    // state in sk_flags[b + 2][warp].
    int64_t dp_tiles;
    float *sk_part;        // [2 * pairs] k-tail slots of 128 x BNP fp32, [BNP/4][128][4]
    float *sk_head;        // [2 * pairs] k-head slots, same layout
    uint32_t *sk_flags;    // [2 * pairs][4]
    uint32_t epoch;
    int sk_mode;           // test hook, as in the single-CTA kernel
};

// kTmaStore: C by TMA stores (else predicated stores, for a C whose rows TMA
// cannot describe; A and B always come by TMA).
template <bool kTmaStore = true>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_relu_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const Params p) {
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
    const uint32_t rank = cluster_ctarank();          // 0: issues the MMAs
    const bool leader = rank == 0;
    const int64_t pair_id = blockIdx.x >> 1;
    const int64_t num_pairs = gridDim.x >> 1;
    const SkShape sk{p.num_tiles, p.dp_tiles, p.num_kb};

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < (uint32_t)kStages; ++s) {
            mbar_init(full_bar(s), 1u);               // the leader's expect_tx arrival
            mbar_init(empty_bar(s), 1u);              // one multicast commit
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1u);
            mbar_init(acce_bar(b), 2u * kEpiWarps);   // both CTAs' epilogue warps
        }
        mbar_init(drain_bar, 1u);
        *abort_flag = 0u;
        fence_mbar_init();
        pdl_launch_dependents();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        if (kTmaStore)
            tma_prefetch_map(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    cluster_sync();          // both CTAs' barriers initialised before any remote signal
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    pdl_wait_primary();      // the previous grid of the stream has completed

    if (warp == 0) {
        // ============================================================ producer
        // Both CTAs: own A rows and B columns of each k block, counted on the
        // leader's full[stage]; the leader also posts the pair's byte count.
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0, parity = 0;
            bool ok = true;
            const int64_t items = sk_num_items(sk, pair_id, num_pairs);
            for (int64_t it = 0; ok && it < items; ++it) {
                int64_t t, mb, nb;
                int kb0, kb1, kind;
                sk_item_at(sk, pair_id, num_pairs, it, t, kb0, kb1, kind);
                tile_coord(t, p.m_tiles, p.n_tiles, p.panel, mb, nb);
                const int m0 = (int)(mb * BMP) + 128 * (int)rank;
                const int n0 = (int)(nb * BNP) + kBHalf * (int)rank;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, p.wait_limit_ns, abort_flag,
                                      kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const bool drop = p.drop_arrive && blockIdx.x == 0 && it == 0 && kb == kb0;
                    if (!drop) {
                        const uint32_t fb = mapa_shared(full_bar(stage), 0);
                        if (leader)
                            mbar_arrive_expect_tx(full_bar(stage), 2 * kStageBytes);
                        tma_load_2d_pair(&tmA, base + kOffA + stage * kATile, fb, kb * BK, m0);
                        const uint32_t bdst = base + kOffB + stage * kBTile;
#pragma unroll
                        for (int j = 0; j < kBHalf / 64; ++j)
                            tma_load_2d_pair(&tmB, bdst + j * kBSlab, fb, n0 + 64 * j, kb * BK);
                        issued |= 1u << stage;
                        parity = (parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == (uint32_t)kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // The leader's full barriers count both CTAs' copies: once its
            // last phases completed, nothing the pair issued is in flight.
            if (leader)
                for (uint32_t s = 0; s < (uint32_t)kStages; ++s)
                    if (issued & (1u << s))
                        wait_drain(full_bar(s), (parity >> s) & 1u, p.wait_limit_ns, abort_flag);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (leader && lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            const int64_t items = sk_num_items(sk, pair_id, num_pairs);
            for (int64_t i = 0; ok && i < items; ++i) {
                int64_t t;
                int kb0, kb1, kind;
                sk_item_at(sk, pair_id, num_pairs, i, t, kb0, kb1, kind);
                const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
                if (!wait_bounded(acce_bar(buf), use ^ 1u, p.wait_limit_ns, abort_flag,
                                  kSiteMmaAccEmpty))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + buf * BNP;
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
                        const uint64_t adesc = make_sdesc_sw128(a + kk * (UK * 2), 16, 1024);
                        const uint64_t bdesc = make_sdesc_sw128(b + kk * (UK * 128), kBSlab, 1024);
                        umma_f16_pair(d, adesc, bdesc, kIdesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit_pair(empty_bar(stage), 0x3);   // both CTAs may refill
                    if (++stage == (uint32_t)kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit_pair(accf_bar(buf), 0x3);          // both CTAs' accumulators ready
            }
            umma_commit_pair(drain_bar, 0x1);
            wait_drain(drain_bar, 0u, p.wait_limit_ns, abort_flag);
        }
    } else {
        // ============================================================ epilogue
        // Both CTAs: rows [128 rank, +128) of the tile from own TMEM -> ReLU
        // -> fp16 -> swizzled staging -> TMA store; then release the
        // accumulator buffer on the leader's acc_empty (remote for rank 1).
        const int ew = warp - 2;                // staging buffer owner 0..3
        const int q = warp & 3;                 // TMEM lanes 32q .. 32q+31
        const int row_in_tile = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t stage_base = base + kOffEpi + (uint32_t)ew * 2u * kEpiBuf;
        uint32_t nstores = 0;
        const int64_t items = sk_num_items(sk, pair_id, num_pairs);
        const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
        // Stream-K: as in the single-CTA kernel, the next pair's published k
        // tail (this CTA's rows) is pre-loaded into the spare TMEM buffer when
        // it is already there once the item before the k head has been read;
        // otherwise the two sides meet through the wait-free exchange.
        int64_t last_t = 0;
        int last_kb0 = 0, last_kb1 = 0, last_kind = kItemFull;
        if (items > 0)
            sk_item_at(sk, pair_id, num_pairs, items - 1, last_t, last_kb0, last_kb1, last_kind);
        const bool head_last = last_kind == kItemPieceIn;
        const uint32_t partner_buf = tmem_base + lane_base + (uint32_t)((items - 2) & 1) * BNP;
        constexpr size_t kSlot = (size_t)BNP * 128;
        uint32_t *const head_cut = p.sk_flags + (blockIdx.x + 2) * 4 + q;
        uint32_t *const tail_cut = p.sk_flags + blockIdx.x * 4 + q;
        const float *const next_tail = p.sk_part + (size_t)(blockIdx.x + 2) * kSlot;
        const float *const prev_head =
            blockIdx.x >= 2 ? p.sk_head + (size_t)(blockIdx.x - 2) * kSlot : nullptr;
        bool preloaded = false;
        auto try_preload = [&]() {
            if (p.sk_mode != 0 || fused::sk_peek(head_cut, lane) != fused::sk_tail_tag(p.epoch))
                return;
            fused::piece_to_tmem<BNP>(next_tail, row_in_tile, partner_buf);
            __syncwarp();
            if (lane == 0)
                *head_cut = 0u;  // consumed
            preloaded = true;
        };
        auto publish = [&](float *slot, uint32_t acc) {
#pragma unroll 1
            for (int c = 0; c < BNP / 32; ++c) {
                uint32_t r[32];
                tmem_ld_x32_sync(acc + 32 * c, r);
                fused::piece_store32(slot, row_in_tile, 32 * c, r);
            }
        };
        // Stores this CTA's 128 rows of tile t from `acc` (+ the TMEM partner
        // buffer when add == 1, + a published piece when add == 2).
        auto store_tile = [&](int64_t t, uint32_t acc, int add, const float *piece) {
            int64_t mb, nb;
            tile_coord(t, p.m_tiles, p.n_tiles, p.panel, mb, nb);
            const int64_t row0 = mb * BMP + 128 * (int64_t)rank + 32 * q;
            const int64_t n0 = nb * BNP;
#pragma unroll 1
            for (int c = 0; c < BNP / 64; ++c) {
                const int64_t col0 = n0 + 64 * c;
                if (row0 >= p.M || col0 >= p.N)
                    continue;  // warp-uniform: nothing of this chunk is in C
                uint32_t r[32], h[32];
                const uint32_t taddr = acc + 64 * c;
                tmem_ld_x32_sync(taddr, r);
                if (add == 1)
                    fused::add_tmem(r, partner_buf + 64 * c);
                else if (add == 2)
                    fused::add_slot32(r, piece, row_in_tile, 64 * c);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    h[j] = relu_pack_half2(r[2 * j], r[2 * j + 1]);
                tmem_ld_x32_sync(taddr + 32, r);
                if (add == 1)
                    fused::add_tmem(r, partner_buf + 64 * c + 32);
                else if (add == 2)
                    fused::add_slot32(r, piece, row_in_tile, 64 * c + 32);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    h[16 + j] = relu_pack_half2(r[2 * j], r[2 * j + 1]);
                if constexpr (kTmaStore) {
                    const uint32_t sb = stage_base + (nstores & 1u) * kEpiBuf;
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
        for (int64_t i = 0; i < items; ++i) {
            int64_t t;
            int kb0, kb1, kind;
            sk_item_at(sk, pair_id, num_pairs, i, t, kb0, kb1, kind);
            const uint32_t buf = (uint32_t)(i & 1), use = (uint32_t)((i >> 1) & 1);
            const bool ok = wait_bounded(accf_bar(buf), use, p.wait_limit_ns, abort_flag,
                                         kSiteEpiAccFull);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after_sync();
            const uint32_t acc = tmem_base + lane_base + buf * BNP;
            if (kind == kItemPieceOut) {
                // k tail of a tile cut with the previous pair: publish it; if
                // that pair's k head was published first, finish the tile here
                if (p.sk_mode == 2)
                    fused::sk_test_delay(200000);
                publish(p.sk_part + (size_t)blockIdx.x * kSlot, acc);
                if (fused::sk_exchange(tail_cut, fused::sk_tail_tag(p.epoch), lane) ==
                    fused::sk_head_tag(p.epoch)) {
                    store_tile(t, acc, 2, prev_head);
                    __syncwarp();
                    if (lane == 0)
                        *tail_cut = 0u;  // consumed
                }
            } else if (kind == kItemPieceIn) {
                // k head of a tile cut with the next pair: add its k tail if
                // it is there; else publish the head and finish only if the
                // tail arrived meanwhile
                if (p.sk_mode == 3)
                    fused::sk_test_delay(200000);
                int add = preloaded ? 1 : 0;
                if (!preloaded) {
                    if (p.sk_mode == 0 &&
                        fused::sk_peek(head_cut, lane) == fused::sk_tail_tag(p.epoch)) {
                        add = 2;
                    } else {
                        publish(p.sk_head + (size_t)blockIdx.x * kSlot, acc);
                        add = fused::sk_exchange(head_cut, fused::sk_head_tag(p.epoch), lane) ==
                                      fused::sk_tail_tag(p.epoch)
                                  ? 2
                                  : -1;  // -1: the next pair finishes the tile
                    }
                }
                if (add >= 0) {
                    store_tile(t, acc, add, next_tail);
                    if (add == 2) {
                        __syncwarp();
                        if (lane == 0)
                            *head_cut = 0u;  // consumed
                    }
                }
            } else {
                store_tile(t, acc, 0, nullptr);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(acce_leader0 + 8u * buf);
            if (head_last && items >= 2 && i == items - 2)
                try_preload();
        }
        if (kTmaStore && lane == 0)
            bulk_wait_group<0>();
    }

    // ---------------------------------------------------------------- teardown
    // Neither CTA leaves while the pair's MMAs may still read its shared
    // memory or signal its barriers; then both free the pair's TMEM.
    __syncwarp();
    tc_fence_before_sync();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace pair
}  // namespace gemmrelu
