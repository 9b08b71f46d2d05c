// gemm_relu_gemv.cuh -- C = fp16(max(A . B, 0)) for M <= 8 (decode-like rows;
// the library routes M <= 4 here by default).
//
// The GEMV pattern of "TileLang CUDA 核心编程模式" section 4: one thread per
// output column keeps an fp32 accumulator in registers while it walks K,
// with the operands staged through shared memory.  With M <= 8 every element
// of B feeds at most eight multiply-adds, so the work is a stream of B
// through HBM and the tensor cores would idle; it runs on the CUDA cores:
//
//   * B (K x N, row-major) is cut into column blocks of 256 and K chunks.  A
//     CTA owns one (column block, K chunk); the K chunks of a column block
//     form a thread-block cluster of up to 8 CTAs.
//   * Lane 0 of warp 0 streams the CTA's 32-row x 256-column boxes of B
//     with TMA into a 4-stage shared-memory ring (evict-first in L2: B is read
//     once), refilling each slot as soon as all warps have released it.
//   * Eight compute warps: lane l owns columns 8l .. 8l+7 of the block (one
//     16-byte shared load per row), warp w rows 4w .. 4w+3 of every stage.
//     Each stage also carries the 8 x 32 box of A for its rows (TMA, zero
//     fill beyond M and K).  Accumulation: fp32 multiply-add straight from
//     the fp16 operands (the mixed-precision FMA of sm_100 and later), so no
//     conversion instructions; it rounds exactly as converting to fp32 and
//     fma.rn.f32 would.
//   * Reduction in a fixed order: the eight warps' partials (through the
//     drained stage buffers), then the cluster's K chunks in rank order
//     through distributed shared memory; ReLU; fp16.
//
// Every sum has a fixed order, so results are the same from run to run.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "gemm_relu_kernels.cuh"

// Stages each CTA asks L2 to fetch before it waits for the previous grid.
#ifndef GEMMRELU_GEMV_PREFETCH
#define GEMMRELU_GEMV_PREFETCH 8
#endif

namespace gemmrelu {
namespace gemv {

constexpr int kCols = 256;          // columns of B per CTA (TMA box width)
constexpr int kRows = 32;           // rows of B per stage (TMA box height)
constexpr int kStages = 4;
constexpr int kWarps = 8;           // all compute; lane 0 of warp 0 also issues the TMA copies
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxCluster = 8;
constexpr int kMaxM = 8;
constexpr uint32_t kBBytes = kCols * kRows * 2;        // 16 KB: [32 k][256 n] fp16
constexpr uint32_t kABytes = kMaxM * kRows * 2;        // 512 B: [8 m][32 k] fp16
constexpr uint32_t kStageBytes = kBBytes + kABytes;    // a multiple of 128
constexpr uint32_t kRing = kStages * kStageBytes;
constexpr uint32_t kOffRed = kRing;                    // cluster buffer: kMaxM x 256 fp32
constexpr uint32_t kRedBytes = kMaxM * kCols * 4;
constexpr uint32_t kOffBar = kOffRed + kRedBytes;
constexpr uint32_t kOffMisc = kOffBar + 2 * kStages * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
static_assert(kWarps * kMaxM * kCols * 4 <= kRing, "warp partials reuse the stage ring");

struct Params {
    uint16_t *C;           // M x N, row-major fp16
    int M, N, K;
    int num_stages;        // ceil(K / kRows)
    int drop_arrive;
    uint64_t wait_limit_ns;
};

// d0 += a * b.lo, d1 += a * b.hi with fp16 a (the low or high half of a2) and
// fp16 pair b2, accumulated in fp32 (mixed-precision FMA of sm_100 and later;
// the fp16 x fp16 product is exact in fp32, so this rounds exactly like
// converting both to fp32 and using fma.rn.f32).
template <bool kHi>
__device__ __forceinline__ void mfma2(float &d0, float &d1, uint32_t a2, uint32_t b2) {
    if constexpr (kHi)
        asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
            "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
            "fma.rn.f32.f16 %0, ah, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
            : "+f"(d0), "+f"(d1)
            : "r"(a2), "r"(b2));
    else
        asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
            "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
            "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, al, bh, %1;\n\t}"
            : "+f"(d0), "+f"(d1)
            : "r"(a2), "r"(b2));
}

__device__ __forceinline__ uint4 ld_shared_v4u(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// One CTA: column block blockIdx.x / csize, K chunk = its cluster rank (the
// stages [rank * S / csize, (rank + 1) * S / csize) of the S 32-row stages).
// MV = rows of accumulators (M rounded up to 1, 2, 4 or 8).
template <int MV>
__global__ void __launch_bounds__(kThreads, 2)
    gemm_relu_gemv_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const Params p, int csize) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kOffBar;
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (kStages + s); };
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + kOffMisc);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int n0 = (int)(blockIdx.x / (unsigned)csize) * kCols;
    const int s0 = (int)(((int64_t)rank * p.num_stages) / csize);
    const int s1 = (int)(((int64_t)(rank + 1) * p.num_stages) / csize);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < (uint32_t)kStages; ++s) {
            mbar_init(full_bar(s), 1u);
            mbar_init(empty_bar(s), (uint32_t)kWarps);
        }
        *abort_flag = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
        pdl_launch_dependents();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        // L2 fetches the first stages while the previous grid finishes (L2
        // is the point of coherence: this moves nothing past the dependence)
        for (int j = s0; j < s1 && j < s0 + GEMMRELU_GEMV_PREFETCH; ++j) {
            tma_prefetch_2d(&tmB, n0, j * kRows);
            tma_prefetch_2d(&tmA, j * kRows, 0);
        }
    }
    __syncthreads();
    pdl_wait_primary();  // the previous grid of the stream has completed

    // TMA issue for the stage s0 + j (lane 0 of warp 0 only); slot j % kStages
    // must have been released by all warps for stage j - kStages.
    const uint64_t stream_once = l2_policy_evict_first();
    uint32_t issued = 0, parity = 0;
    auto issue = [&](int j) -> bool {
        const uint32_t slot = (uint32_t)(j % kStages);
        const uint32_t phase = (uint32_t)((j / kStages) & 1);
        if (!wait_bounded(empty_bar(slot), phase ^ 1u, p.wait_limit_ns, abort_flag,
                          kSiteProducerEmpty))
            return false;
        if (p.drop_arrive && blockIdx.x == 0 && j == 0)
            return true;  // test hook: this stage never arrives
        const uint32_t fb = full_bar(slot);
        const uint32_t dst = base + slot * kStageBytes;
        const int k0 = (s0 + j) * kRows;
        mbar_arrive_expect_tx(fb, kStageBytes);
        tma_load_2d_hint(&tmB, dst, fb, n0, k0, stream_once);
        tma_load_2d(&tmA, dst + kBBytes, fb, k0, 0);
        issued |= 1u << slot;
        parity = (parity & ~(1u << slot)) | (phase << slot);
        return true;
    };
    const int n_st = s1 - s0;
    const bool producer = threadIdx.x == 0;
    bool feeding = true;
    if (producer)
        for (int j = 0; feeding && j < kStages - 1 && j < n_st; ++j)
            feeding = issue(j);

    float2 acc[MV][4];  // columns 8l + 2j, 8l + 2j + 1
#pragma unroll
    for (int m = 0; m < MV; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[m][j] = make_float2(0.0f, 0.0f);
    // rows 4w .. 4w+3 of each stage; columns 8l .. 8l+7 of the block
    const uint32_t b_off = (uint32_t)(4 * warp) * (kCols * 2) + (uint32_t)lane * 16;
    const uint32_t a_off = kBBytes + (uint32_t)(4 * warp) * 2;
    for (int i = 0; i < n_st; ++i) {
        if (producer && feeding && i + kStages - 1 < n_st)
            feeding = issue(i + kStages - 1);
        const uint32_t slot = (uint32_t)(i % kStages);
        const uint32_t phase = (uint32_t)((i / kStages) & 1);
        const bool ok = wait_bounded(full_bar(slot), phase, p.wait_limit_ns, abort_flag,
                                     kSiteMmaFull);
        if (!__all_sync(0xffffffffu, ok))
            break;
        const uint32_t st = base + slot * kStageBytes;
#pragma unroll
        for (int rp = 0; rp < 2; ++rp) {
            // A[m][4w + 2rp] (low half) and A[m][4w + 2rp + 1] (high half)
            uint32_t a2[MV];
#pragma unroll
            for (int m = 0; m < MV; ++m)
                a2[m] = ld_shared_b32(st + a_off + (uint32_t)m * (kRows * 2) + 4u * rp);
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = 2 * rp + rr;
                const uint4 bv = ld_shared_v4u(st + b_off + (uint32_t)r * (kCols * 2));
                const uint32_t b[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int m = 0; m < MV; ++m)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (rr)
                            mfma2<true>(acc[m][j].x, acc[m][j].y, a2[m], b[j]);
                        else
                            mfma2<false>(acc[m][j].x, acc[m][j].y, a2[m], b[j]);
                    }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty_bar(slot));
    }
    // every copy issued must have landed before the ring is reused
    if (producer)
        for (uint32_t s = 0; s < (uint32_t)kStages; ++s)
            if (issued & (1u << s))
                wait_drain(full_bar(s), (parity >> s) & 1u, p.wait_limit_ns, abort_flag);

    // ---------------------------------------------------------------- reduction
    __syncthreads();  // ring quiescent: every copy consumed (or drained after a timeout)
    // warp partials into the ring: part[w][m][column]
#pragma unroll
    for (int m = 0; m < MV; ++m) {
        const uint32_t a = base + ((uint32_t)(warp * MV + m) * kCols + 8u * lane) * 4u;
        st_shared_v4(a, __float_as_uint(acc[m][0].x), __float_as_uint(acc[m][0].y),
                     __float_as_uint(acc[m][1].x), __float_as_uint(acc[m][1].y));
        st_shared_v4(a + 16u, __float_as_uint(acc[m][2].x), __float_as_uint(acc[m][2].y),
                     __float_as_uint(acc[m][3].x), __float_as_uint(acc[m][3].y));
    }
    __syncthreads();
    // column t: the warps' partials in order w = 0..7, then to the CTA of the
    // cluster that owns column t (kCols / csize columns each), slot = rank
    const uint32_t per_owner = (uint32_t)(kCols / csize);
    const uint32_t red = base + kOffRed;
    if (threadIdx.x < kCols) {
        const uint32_t t = threadIdx.x;
        const uint32_t owner = t / per_owner, c = t % per_owner;
#pragma unroll
        for (int m = 0; m < MV; ++m) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                v += __uint_as_float(ld_shared_b32(base + ((uint32_t)(w * MV + m) * kCols + t) * 4u));
            st_cluster_f32(mapa_shared(red + ((rank * MV + (uint32_t)m) * per_owner + c) * 4u, owner),
                           v);
        }
    }
    cluster_sync();  // every CTA's column partials delivered; no remote access after this
    // this CTA's columns: the K chunks in rank order, then ReLU and fp16
    for (uint32_t idx = threadIdx.x; idx < (uint32_t)MV * per_owner; idx += kThreads) {
        const uint32_t m = idx / per_owner, c = idx % per_owner;
        float v = 0.0f;
        for (int r = 0; r < csize; ++r)
            v += __uint_as_float(ld_shared_b32(red + (((uint32_t)r * MV + m) * per_owner + c) * 4u));
        const int64_t col = (int64_t)n0 + rank * per_owner + c;
        if ((int)m < p.M && col < p.N)
            p.C[(int64_t)m * p.N + col] = (uint16_t)(relu_pack_half2(__float_as_uint(v), 0u) & 0xffffu);
    }
}

}  // namespace gemv
}  // namespace gemmrelu
