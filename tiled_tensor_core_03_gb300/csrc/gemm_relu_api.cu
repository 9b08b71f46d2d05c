// gemm_relu_api.cu -- the C ABI of libgemmrelu.so (declared in gemm_relu.h).
//
// Host side only: argument checks, choice of operand path, TMA tensor-map
// encoding (CUDA driver entry point fetched through the runtime, so the
// library needs no link against libcuda), launch configuration and the
// device status word.  Every arithmetic step runs in the kernels of
// gemm_relu_kernels.cuh and gemm_relu_splitk.cuh; there is no host or library
// fallback.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>
#include <random>
#include <utility>

#include "gemm_relu.h"
#include "flash_attention.h"
#include "gemm_relu_kernels.cuh"
#include "gemm_relu_splitk.cuh"
#include "gemm_relu_2sm.cuh"
#include "gemm_relu_gemv.cuh"
#include "flash_attention.cuh"
#include "gemm_relu_stage.cuh"

namespace {

using gemmrelu::tile_coord;

constexpr int64_t kMaxDim = 0x7fffffff;
#ifndef GEMMRELU_SPLIT_MAJOR
#define GEMMRELU_SPLIT_MAJOR 1
#endif
constexpr int64_t kPanelBytes = 32ll << 20;         // A rows per rasteriser panel, in bytes
constexpr int kSplitMajor = GEMMRELU_SPLIT_MAJOR;  // split-K work-unit order
constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------- test hooks
std::atomic<int> g_drop_arrive{0};
std::atomic<int64_t> g_wait_limit_ns{0};
std::atomic<int> g_force_kernel{0};   // 0 auto, 1 one CTA x 256, 2 one CTA x 128, 3 CTA pair,
                                      // 4 GEMV (M <= 8)
std::atomic<int> g_force_split{0};    // 0 auto, 1 two-stage split-K form only
std::atomic<int> g_panel_rows{0};     // 0 the default panel, else output rows per panel
std::atomic<int> g_sk_mode{0};        // stream-K fix-up test mode (0 normal)
std::atomic<int> g_sk_pieces{0};      // sub-wave pieces per tile (0: the library's choice)
// Starts from a value drawn per process, so that state words a stream-K call
// of another process left behind in reused device memory are unlikely to
// carry the tag of one of this process's calls.
std::atomic<uint32_t> g_epoch{(uint32_t)std::random_device{}()};

// Stream-K calls are told apart by an epoch below 2^30 (the fix-up tags its
// state words with epoch * 4 + 1 or + 2), never 0; the side that finishes a
// cut tile resets its state word to 0.
uint32_t next_epoch() {
    for (;;) {
        const uint32_t e = (++g_epoch) & 0x3fffffffu;
        if (e)
            return e;
    }
}

// Rasteriser panel height in output rows for a contraction of length K.
// A panel's A rows (rows x K fp16) are read while the panel sweeps every
// column of B, so they should stay in L2 for the whole sweep while B
// streams past: panels are as tall as fits in 32 MiB (a quarter of L2).
// B is then read from DRAM about once per panel.  Measured on GB300 (CTA-pair
// kernel, 256-row panel steps): 8192 x 8192 x 4096 reads 244 MB of DRAM with
// 4096-row panels against 495 MB with 1024-row ones, and runs 3.5% faster;
// 16384 x 16384 x 4096 and 4096 x 16384 x 4096 6% faster, 8192^3 and 6144^3
// 2% faster with 2048-row panels; at 4096^3 (everything fits in L2) the
// height makes no difference.
int64_t panel_rows_for(int64_t K) {
    const int rows = g_panel_rows.load();
    if (rows > 0)
        return rows;
    const int64_t fit = (int64_t)(kPanelBytes / (2 * std::max<int64_t>(K, 1)));
    return std::max<int64_t>(256, fit / 256 * 256);
}

// The same panel in tiles of `tile_rows` output rows.
int panel_tiles(int tile_rows, int64_t K) {
    const int64_t tiles = panel_rows_for(K) / tile_rows;
    return (int)std::max<int64_t>(1, std::min<int64_t>(tiles, kMaxDim));
}

uint64_t wait_limit_ns() {
    const int64_t v = g_wait_limit_ns.load();
    return v > 0 ? (uint64_t)v : kDefaultWaitLimitNs;
}

// ---------------------------------------------------------------- per device
struct DeviceState {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    bool attr_fused[6] = {false, false, false, false, false, false};
    bool attr_split[4] = {false, false, false, false};
    bool attr_split_cluster[4] = {false, false, false, false};
    int split_pairs[4] = {};  // max resident CTA pairs of the cluster form, per bms index
    bool attr_pair = false;
    bool attr_pair_pred = false;
    bool attr_gemv[4] = {false, false, false, false};
    bool attr_attn[2] = {false, false};
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

int current_device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return GEMMRELU_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &s = g_dev[dev];
    if (!s.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMMRELU_ERR_CUDA;
        s.supported = (major == 10 && minor == 3);
        s.sms = sms;
        s.probed = true;
    }
    *out = &s;
    return s.supported ? GEMMRELU_OK : GEMMRELU_ERR_UNSUPPORTED_DEVICE;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major fp16 matrix rows x cols (cols contiguous), box box_cols x box_rows,
// 128-byte swizzle (or none), zero fill outside the matrix.
bool make_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
              int64_t pitch = 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(pitch > 0 ? pitch : cols) * 2};  // row pitch, bytes
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows res, res + 8, res + 16, ... of a row-major fp16 matrix rows x cols
// whose pitch need not be a multiple of 16 bytes, as a 2-D tensor for the
// predicated-load kernel (see gemmrelu::fused::RowMaps): base = the first
// such row's start rounded down to 16 bytes, row stride 8 rows (16 * cols
// bytes), cols + off / 2 elements per row (off = the start's byte offset in
// its 16-byte block), no swizzle, zero fill outside.  Needs res < rows.
bool make_row_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, int64_t res,
                  uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const uintptr_t start = reinterpret_cast<uintptr_t>(ptr) + (uintptr_t)(2 * res * cols);
    const uintptr_t base = start & ~(uintptr_t)15;
    cuuint64_t dims[2] = {(cuuint64_t)(cols + (int64_t)(start - base) / 2),
                          (cuuint64_t)((rows - res + 7) / 8)};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 16};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, reinterpret_cast<void *>(base), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- argument checks
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_args(const void *A, const void *B, const void *C, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMMRELU_ERR_INVALID_ARG;
    if (M == 0 || N == 0)
        return GEMMRELU_OK;
    if (!C || !aligned(C, 2))
        return GEMMRELU_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B || !aligned(A, 2) || !aligned(B, 2)))
        return GEMMRELU_ERR_INVALID_ARG;
    return GEMMRELU_OK;
}

// TMA can describe a row-major fp16 matrix when its base is 16-byte aligned
// and its row pitch (cols * 2 bytes) is a multiple of 16 bytes.
bool tma_ok(const void *p, int64_t cols) { return aligned(p, 16) && (cols % 8) == 0; }

int fused_path(const void *A, const void *B, const void *C, int64_t M, int64_t N, int64_t K) {
    if (check_args(A, B, C, M, N, K) != GEMMRELU_OK)
        return -1;
    if (M == 0 || N == 0 || K == 0)
        return 0;
    return (tma_ok(A, K) && tma_ok(B, N) && tma_ok(C, N)) ? 1 : 2;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? GEMMRELU_OK : GEMMRELU_ERR_LAUNCH; }

template <typename Kern>
bool ensure_smem_attr(bool &done, Kern kernel, uint32_t bytes) {
    if (done)
        return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
        return false;
    done = true;
    return true;
}

#ifndef GEMMRELU_PDL
#define GEMMRELU_PDL 1
#endif

// Every kernel of this library is launched through here, with programmatic
// stream serialisation: it may become resident while the previous grid of
// the stream finishes, overlapping its start-up (barrier set-up, TMEM
// allocation, descriptor prefetch) with that grid's tail; the kernel waits
// for the previous grid (griddepcontrol.wait) before it touches global
// memory.  `cooperative` guarantees co-residency of all CTAs (stream-K);
// cluster_x > 1 sets a cluster shape at launch.
template <typename... KArgs, typename... Args>
int launch_kernel(void (*kern)(KArgs...), unsigned grid, unsigned block, uint32_t smem,
                  cudaStream_t stream, bool cooperative, unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    unsigned n = 0;
    if (GEMMRELU_PDL) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return launch_status(cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...));
}

int zero_fill(void *C, int64_t M, int64_t N, cudaStream_t stream) {
    return launch_status(cudaMemsetAsync(C, 0, (size_t)M * (size_t)N * 2, stream));
}

// ---------------------------------------------------------------- fused launch
#ifndef GEMMRELU_FUSED_BN
#define GEMMRELU_FUSED_BN 0       // 0: choose per shape; 128 or 256: force
#endif

// Tile width of the fused kernel: 256 unless 128-wide tiles fill the SMs in
// fewer weighted waves.  Measured on GB300, a 128-wide tile costs about 0.7 of
// a 256-wide one (its MMAs are bound by shared-memory bandwidth), so 128 only
// wins when it turns a partial wave into a full one, as at 1024^3.
int fused_bn(int64_t M, int64_t N, int sms) {
    if (GEMMRELU_FUSED_BN == 128 || GEMMRELU_FUSED_BN == 256)
        return GEMMRELU_FUSED_BN;
    if (g_force_kernel.load() == 1)
        return 256;
    if (g_force_kernel.load() == 2)
        return 128;
    const int64_t mt = (M + 127) / 128;
    const int64_t w256 = (mt * ((N + 255) / 256) + sms - 1) / sms;
    const int64_t w128 = (mt * ((N + 127) / 128) + sms - 1) / sms;
    return (double)w128 * 0.7 < (double)w256 ? 128 : 256;
}

template <bool kTma, int kBN, bool kTmaStore = kTma>
int launch_fused_bn(const CUtensorMap &mA, const CUtensorMap &mB, const CUtensorMap &mC,
                    const gemmrelu::fused::Params &p, const gemmrelu::fused::MapsFor<kTma> &rm,
                    int64_t grid, cudaStream_t stream, bool &attr_done) {
    namespace F = gemmrelu::fused;
    auto kern = F::gemm_relu_fused_kernel<kTma, kBN, kTmaStore>;
    constexpr uint32_t smem = F::Tile<kBN, kTma>::kSmemBytes;
    if (!ensure_smem_attr(attr_done, kern, smem))
        return GEMMRELU_ERR_LAUNCH;
    // (stream-K needs no co-residency: its fix-up never waits for another CTA)
    return launch_kernel(kern, (unsigned)grid, F::Roles<kTma>::kThreads, smem, stream,
                         false, 1, mA, mB, mC, p, rm);
}

// Stream-K part of a fused launch: dp_tiles < num_tiles, with its workspace.
struct StreamK {
    int64_t dp_tiles = -1;     // -1: plain data-parallel launch
    int64_t ctas = 0;          // grid of a stream-K launch
    float *part = nullptr;     // k-tail slots
    float *head = nullptr;     // k-head slots
    uint32_t *flags = nullptr; // fix-up state words
    uint32_t epoch = 0;
};

// ---------------------------------------------------------------- CTA-pair launch
// 256 x 256 tiles on CTA pairs (2-SM MMA).  A and B by TMA (row pitches lda,
// ldb elements: K and N for the caller's own operands, wider for staged
// copies); C by TMA stores when its rows allow, else predicated stores.
int launch_pair(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                cudaStream_t stream, DeviceState *ds, const StreamK &sk = StreamK(),
                int64_t lda = 0, int64_t ldb = 0) {
    namespace P = gemmrelu::pair;
    namespace F = gemmrelu::fused;
    P::Params p{};
    p.C = static_cast<uint16_t *>(C);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.num_kb = (int)((K + P::BK - 1) / P::BK);
    p.m_tiles = (M + P::BMP - 1) / P::BMP;
    p.n_tiles = (N + P::BNP - 1) / P::BNP;
    p.num_tiles = p.m_tiles * p.n_tiles;
    p.panel = panel_tiles(P::BMP, K);
    p.drop_arrive = g_drop_arrive.load();
    p.wait_limit_ns = wait_limit_ns();
    p.dp_tiles = sk.dp_tiles >= 0 ? sk.dp_tiles : p.num_tiles;
    p.sk_part = sk.part;
    p.sk_head = sk.head;
    p.sk_flags = sk.flags;
    p.epoch = sk.epoch;
    p.sk_mode = g_sk_mode.load();
    const bool c_tma = tma_ok(C, N);
    CUtensorMap mA, mB, mC;
    std::memset(&mC, 0, sizeof(mC));
    if (!make_map(&mA, A, M, K, F::BK, F::BM, CU_TENSOR_MAP_SWIZZLE_128B, lda) ||
        !make_map(&mB, B, K, N, 64, F::BK, CU_TENSOR_MAP_SWIZZLE_128B, ldb) ||
        (c_tma && !make_map(&mC, C, M, N, 64, 32)))
        return GEMMRELU_ERR_LAUNCH;
    const int64_t pairs = std::min<int64_t>(p.num_tiles, ds->sms / 2);
    // (stream-K needs no co-residency: its fix-up never waits for another CTA)
    if (c_tma) {
        if (!ensure_smem_attr(ds->attr_pair, P::gemm_relu_pair_kernel<true>, P::kSmemBytes))
            return GEMMRELU_ERR_LAUNCH;
        return launch_kernel(P::gemm_relu_pair_kernel<true>, (unsigned)(2 * pairs), P::kThreads,
                             P::kSmemBytes, stream, false, 1, mA, mB, mC, p);
    }
    if (!ensure_smem_attr(ds->attr_pair_pred, P::gemm_relu_pair_kernel<false>, P::kSmemBytes))
        return GEMMRELU_ERR_LAUNCH;
    return launch_kernel(P::gemm_relu_pair_kernel<false>, (unsigned)(2 * pairs), P::kThreads,
                         P::kSmemBytes, stream, false, 1, mA, mB, mC, p);
}

// ---------------------------------------------------------------- GEMV (M <= 8)
namespace V = gemmrelu::gemv;

// Whether a plain (unsplit, not stream-K) launch runs the GEMV kernel: TMA-
// capable A and B and at most four rows (eight when forced).  Measured on
// GB300 at N = K = 8192: M = 1, 2, 4 stream B at 5.3, 5.1, 4.9 TB/s; at M = 8
// the multiply-adds, not HBM, set the pace (37 us) and the tensor-core split
// below is faster (29 us).
constexpr int64_t kGemvMaxM = 4;

bool use_skinny_split(const void *A, const void *B, int64_t M, int64_t N, int64_t K, int sms);

// Decode-like rows.  M <= 2: the GEMV kernel.  M = 3 or 4: the GEMV kernel's
// four accumulator rows cost issue slots, and the split-K pair form with
// S = 2 streams B faster when its pairs (one per 128 columns) fit in one
// wave (measured 4096^2: 11.3 vs 12.3 us; 8192^2: 22.6 vs 23.5 us); with
// more columns the GEMV kernel stays ahead (16384^2: 78.6 vs 84.2 us).
bool use_gemv(const void *A, const void *B, int64_t M, int64_t N, int64_t K, int sms) {
    const int force = g_force_kernel.load();
    if (force != 0 && force != 4)
        return false;
    if (M > (force == 4 ? (int64_t)V::kMaxM : kGemvMaxM) || !tma_ok(A, K) || !tma_ok(B, N))
        return false;
    if (force == 4 || M <= 2)
        return true;
    const bool split_one_wave = 2 * ((N + 127) / 128) <= (int64_t)sms &&
                                use_skinny_split(A, B, M, N, K, sms);
    return !split_one_wave;
}

// K chunks per column block (the cluster size): doubled while the grid stays
// within two CTAs per SM and every chunk keeps at least four 32-row stages.
int gemv_csize(int64_t N, int64_t K, int sms) {
    const int64_t blocks = (N + V::kCols - 1) / V::kCols;
    const int64_t stages = (K + V::kRows - 1) / V::kRows;
    int c = 1;
    while (c < V::kMaxCluster && blocks * c * 2 <= 2 * (int64_t)sms && stages >= (int64_t)c * 2 * 4)
        c *= 2;
    return c;
}

template <int MV>
int launch_gemv_mv(const CUtensorMap &mA, const CUtensorMap &mB, const V::Params &p, int csize,
                   int64_t blocks, cudaStream_t stream, bool &attr_done) {
    auto kern = V::gemm_relu_gemv_kernel<MV>;
    if (!ensure_smem_attr(attr_done, kern, V::kSmemBytes))
        return GEMMRELU_ERR_LAUNCH;
    return launch_kernel(kern, (unsigned)(blocks * csize), V::kThreads, V::kSmemBytes, stream,
                         false, (unsigned)csize, mA, mB, p, csize);
}

int launch_gemv(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                cudaStream_t stream, DeviceState *ds) {
    V::Params p{};
    p.C = static_cast<uint16_t *>(C);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.num_stages = (int)((K + V::kRows - 1) / V::kRows);
    p.drop_arrive = g_drop_arrive.load();
    p.wait_limit_ns = wait_limit_ns();
    CUtensorMap mA, mB;
    if (!make_map(&mA, A, M, K, V::kRows, V::kMaxM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mB, B, K, N, V::kCols, V::kRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return GEMMRELU_ERR_LAUNCH;
    const int csize = gemv_csize(N, K, ds->sms);
    const int64_t blocks = (N + V::kCols - 1) / V::kCols;
    if (M <= 1)
        return launch_gemv_mv<1>(mA, mB, p, csize, blocks, stream, ds->attr_gemv[0]);
    if (M <= 2)
        return launch_gemv_mv<2>(mA, mB, p, csize, blocks, stream, ds->attr_gemv[1]);
    if (M <= 4)
        return launch_gemv_mv<4>(mA, mB, p, csize, blocks, stream, ds->attr_gemv[2]);
    return launch_gemv_mv<8>(mA, mB, p, csize, blocks, stream, ds->attr_gemv[3]);
}

// Whether gemm_relu_f16 runs the CTA-pair kernel: TMA operands, at least one
// full 256 x 256 tile, more 128 x 128 tiles than SMs, and no more weighted
// waves than the single-CTA choice (a 256 x 256 pair tile does the work of
// two 128 x 256 tiles on two SMs).  When one wave of 128 x 128 single-CTA
// tiles covers the output, it spreads the work over up to four times as
// many SMs as the pair tiles: measured faster wherever it fits (GB300, us,
// pair -> 128 x 128: 1024^3 9.75 -> 8.65, 1024 x 1024 x 4096 22.4 -> 19.6,
// 1536^3 12.1 -> 11.1, 1920 x 1280 x 1024 10.4 -> 9.2), while at 2048^3, two
// waves of them, the pair stays ahead (15.9 against 20.5).
bool use_pair(int64_t M, int64_t N, int sms, int path) {
    const int force = g_force_kernel.load();
    if (force == 3)
        return path == 1;
    if (force == 1 || force == 2)
        return false;
    if (path != 1 || M < 256 || N < 256 || sms < 2)
        return false;
    if (((M + 127) / 128) * ((N + 127) / 128) <= sms)
        return false;
    const int64_t pair_waves = ((M + 255) / 256 * ((N + 255) / 256) + sms / 2 - 1) / (sms / 2);
    const int64_t one_waves = ((M + 127) / 128 * ((N + 255) / 256) + sms - 1) / sms;
    return pair_waves <= one_waves;
}

int launch_skinny_split(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream, DeviceState *ds);
// The kernel gemm_relu_f16 runs for these arguments (a GEMMRELU_KERNEL_*
// code; 0: nothing to launch, -1: invalid arguments).  launch_fused routes by
// this same function.
int kernel_for(const void *A, const void *B, const void *C, int64_t M, int64_t N, int64_t K,
               int sms) {
    const int path = fused_path(A, B, C, M, N, K);
    if (path <= 0)
        return path;
    if (use_gemv(A, B, M, N, K, sms))
        return GEMMRELU_KERNEL_GEMV;
    if (use_skinny_split(A, B, M, N, K, sms))
        return GEMMRELU_KERNEL_SPLITK_PAIR;
    if (use_pair(M, N, sms, path))
        return GEMMRELU_KERNEL_PAIR;
    if (path == 2)
        return GEMMRELU_KERNEL_PREDICATED;
    return fused_bn(M, N, sms) == 256 ? GEMMRELU_KERNEL_ONE_CTA_256 : GEMMRELU_KERNEL_ONE_CTA_128;
}

// The single-CTA kernel.  tma_loads: A and B by TMA with row pitches lda,
// ldb (elements), C by TMA stores when its rows allow, else predicated
// stores; otherwise the predicated-load kernel (pitches K and N).
int launch_single_cta(const void *A, int64_t lda, const void *B, int64_t ldb, void *C, int64_t M,
                      int64_t N, int64_t K, bool tma_loads, cudaStream_t stream, DeviceState *ds,
                      const StreamK &sk) {
    namespace F = gemmrelu::fused;
    F::Params p{};
    p.A = static_cast<const uint16_t *>(A);
    p.B = static_cast<const uint16_t *>(B);
    p.C = static_cast<uint16_t *>(C);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.num_kb = (int)((K + F::BK - 1) / F::BK);
    // The predicated-load producer is laid out for 128 x 128 tiles.
    const int bn = tma_loads ? fused_bn(M, N, ds->sms) : 128;
    p.m_tiles = (M + F::BM - 1) / F::BM;
    p.n_tiles = (N + bn - 1) / bn;
    p.num_tiles = p.m_tiles * p.n_tiles;
    p.panel = panel_tiles(F::BM, K);
    p.drop_arrive = g_drop_arrive.load();
    p.wait_limit_ns = wait_limit_ns();
    p.dp_tiles = sk.dp_tiles >= 0 ? sk.dp_tiles : p.num_tiles;
    p.sk_part = sk.part;
    p.sk_head = sk.head;
    p.sk_flags = sk.flags;
    p.epoch = sk.epoch;
    p.sk_mode = g_sk_mode.load();
    // persistent grid: one CTA per tile up to one per SM; a stream-K launch
    // has its plan's grid (one CTA per k range)
    const int64_t grid = sk.dp_tiles >= 0 ? sk.ctas : std::min<int64_t>(p.num_tiles, ds->sms);
    CUtensorMap mA, mB, mC;
    std::memset(&mA, 0, sizeof(mA));
    std::memset(&mB, 0, sizeof(mB));
    std::memset(&mC, 0, sizeof(mC));
    if (tma_loads) {
        const bool c_tma = tma_ok(C, N);
        if (!make_map(&mA, A, M, K, F::BK, F::BM, CU_TENSOR_MAP_SWIZZLE_128B, lda) ||
            !make_map(&mB, B, K, N, 64, F::BK, CU_TENSOR_MAP_SWIZZLE_128B, ldb) ||
            (c_tma && !make_map(&mC, C, M, N, 64, 32)))
            return GEMMRELU_ERR_LAUNCH;
        const F::NoMaps none{};
        if (bn == 256)
            return c_tma ? launch_fused_bn<true, 256, true>(mA, mB, mC, p, none, grid, stream,
                                                            ds->attr_fused[0])
                         : launch_fused_bn<true, 256, false>(mA, mB, mC, p, none, grid, stream,
                                                             ds->attr_fused[4]);
        return c_tma ? launch_fused_bn<true, 128, true>(mA, mB, mC, p, none, grid, stream,
                                                        ds->attr_fused[2])
                     : launch_fused_bn<true, 128, false>(mA, mB, mC, p, none, grid, stream,
                                                         ds->attr_fused[5]);
    }
    // predicated-load kernel: one tensor map per row residue modulo 8 of A and B
    F::RowMaps rm;
    std::memset(&rm, 0, sizeof(rm));
    for (int r = 0; r < 8; ++r) {
        if ((r < M && !make_row_map(&rm.a[r], A, M, K, r, F::BK + 8, 16)) ||
            (r < K && !make_row_map(&rm.b[r], B, K, N, r, F::Tile<128, false>::BN + 8, 8)))
            return GEMMRELU_ERR_LAUNCH;
    }
    return launch_fused_bn<false, 128>(mA, mB, mC, p, rm, grid, stream, ds->attr_fused[3]);
}

int launch_fused(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                 cudaStream_t stream, DeviceState *ds, const StreamK &sk = StreamK()) {
    const int path = fused_path(A, B, C, M, N, K);
    if (sk.dp_tiles < 0) {
        switch (kernel_for(A, B, C, M, N, K, ds->sms)) {
        case GEMMRELU_KERNEL_GEMV:
            return launch_gemv(A, B, C, M, N, K, stream, ds);
        case GEMMRELU_KERNEL_SPLITK_PAIR:
            return launch_skinny_split(A, B, C, M, N, K, stream, ds);
        case GEMMRELU_KERNEL_PAIR:
            return launch_pair(A, B, C, M, N, K, stream, ds);
        default:
            break;  // one of the single-CTA kernels, below
        }
    }
    return launch_single_cta(A, K, B, N, C, M, N, K, path == 1, stream, ds, sk);
}

// ---------------------------------------------------------------- stream-K plan
// TMA path only.  When a shape's tiles do not fill a whole number of waves,
// all full waves but the last run data-parallel and the rest is spread
// evenly over the workers (CTA pairs for the pair kernel, CTAs for the
// single-CTA kernel).  The fix-up of the cut tiles (fp32 pieces through L2,
// published after their last MMA) costs a roughly fixed 12-14 us a launch on
// GB300, so this applies only when the plain schedule's partial last wave
// idles longer than that: (ceil(W) - W) * k blocks >= 40 for W = tiles /
// workers.  Measured (CTA pairs, CUDA-graph replay, us, plain / stream-K):
// 2304^2 x 4096 (W 1.07) 41.4 / 35.8, 2560^2 x 4096 (W 1.32) 42.4 / 39.5,
// 4096^3 (W 3.37) 82.0 / 81.7; and where the rule declines: 2304^2 x 1024
// 15.9 / 21.5, 3072^3 (W 1.9) 35.1 / 41.8, 4096^2 x 2048 44.7 / 47.1,
// 4608^2 x 2048 54.4 / 56.5.
//
// With fewer single-CTA tiles than SMs (a partial first wave: small output,
// long K), each tile's k blocks are cut into `pieces` equal ranges on
// pieces * T <= SMs CTAs, pieces = nkb / 128 + 1 clamped to [2, 8] (ranges of
// about 64 to 128 k blocks).  This applies to the single-CTA kernel's shapes
// with M > 64 (fewer rows go to the split-K and GEMV kernels) when the ranges
// come out at least kSkMinSaved k blocks of a 128-column tile shorter than a
// tile, and when an operand that several tiles share fits in half of L2.
// Measured on GB300 (us, plain / 2 / 3 / 4 / 6 pieces): each cut adds a few
// microseconds of fp32 piece traffic through L2 after the last MMA, worth
// some 20 to 40 k blocks of MMA, so short ranges lose (1024^3 on 128 x 128
// tiles 8.6 / 12.0; 200 x 3000 x 2048 12.7 / 14.2; 128 x 4096 x 4096
// 19.3 / 17.4 / 20.4 / 24.4; 128 x 4096 x 8192 33.6 / 24.9 / 26.4 / 29.4) and
// long ones gain (128 x 2048 x 16384 61.9 / 38.3 / 33.6 / 33.8 / 39.2;
// 100 x 1024 x 32768 118.8 / 66.5 / 52.1 / 46.9 / 46.8).  Tiles cut at
// different k offsets read a shared operand at different times, and a large
// one is re-read from DRAM (192 x 6400 x 8192, a 105 MB B shared by two rows
// of tiles: 34.9 -> 45.1 us with 100 tiles spread over 152 CTAs), which also
// lost on an HBM-bound shape (128 x 12800 x 8192: 40.9 -> 47.6 us).
struct SkPlan {
    bool pair = false;
    int64_t dp_tiles = -1;     // -1: no stream-K part
    int64_t ctas = 0;          // grid, and workspace slots (one per CTA)
};

constexpr int64_t kSkMinSaved = 32;
constexpr int64_t kSkMaxSharedBytes = 64ll << 20;

// Multi-wave schedules: worth it when the partial last wave leaves idle at
// least this many k blocks' worth of each worker's time (the fraction of a
// wave left idle, times the k blocks of a tile).
constexpr int64_t kSkMinIdleKb = 40;

bool multiwave_worth_it(int64_t T, int64_t G, int64_t nkb) {
    if (T <= G || T % G == 0)
        return false;
    return (G - T % G) * nkb >= kSkMinIdleKb * G;   // (ceil(T / G) - T / G) * nkb >= 40
}

SkPlan streamk_plan(int64_t M, int64_t N, int64_t K, int path, int sms) {
    namespace F = gemmrelu::fused;
    SkPlan plan;
    if (M <= V::kMaxM || path != 1)
        return plan;  // decode-like rows: the GEMV kernel (or the plain one) serves them
    const int64_t nkb = (K + F::BK - 1) / F::BK;
    if (use_pair(M, N, sms, 1)) {
        const int64_t T = ((M + 255) / 256) * ((N + 255) / 256);
        const int64_t G = std::min<int64_t>(T, sms / 2);
        plan.pair = true;
        plan.ctas = 2 * G;
        if (multiwave_worth_it(T, G, nkb))
            plan.dp_tiles = (T / G - 1) * G;
        return plan;
    }
    const int bn = fused_bn(M, N, sms);
    const int64_t m_tiles = (M + F::BM - 1) / F::BM, n_tiles = (N + bn - 1) / bn;
    const int64_t T = m_tiles * n_tiles;
    if (T >= sms) {
        if (bn == 256 && multiwave_worth_it(T, sms, nkb)) {
            plan.dp_tiles = (T / sms - 1) * sms;
            plan.ctas = sms;
        }
        return plan;
    }
    const int64_t pieces = g_sk_pieces.load() > 0
                               ? g_sk_pieces.load()
                               : std::min<int64_t>({std::max<int64_t>(nkb / 128 + 1, 2), 8,
                                                    sms / std::max<int64_t>(T, 1)});
    const int64_t G = pieces * T;
    if (M <= 64 || pieces < 2 || G > sms)
        return plan;
    const int64_t shared_bytes = (m_tiles > 1 ? 2 * K * N : 0) + (n_tiles > 1 ? 2 * M * K : 0);
    const int64_t longest = (nkb + pieces - 1) / pieces;
    if (shared_bytes > kSkMaxSharedBytes || (nkb - longest) * (bn / 128) < kSkMinSaved)
        return plan;
    plan.dp_tiles = 0;
    plan.ctas = G;
    return plan;
}

// Both kernels' slots hold 128 rows x 256 fp32 columns, plus 4 flags.
constexpr size_t kSkSlotBytes = (size_t)256 * 128 * 4;
size_t streamk_bytes(int64_t ctas) {
    return 2 * (size_t)ctas * kSkSlotBytes + (size_t)ctas * 4 * 4;
}

// ---------------------------------------------------------------- staged operands
// Operands whose rows TMA cannot describe, copied once into aligned rows in
// the caller's workspace (see gemm_relu_stage.cuh): A (M x K) when its pitch
// or base is not 16-byte aligned, B (K x N) likewise, each at a 256-byte
// boundary with its pitch rounded up to 8 elements.  The stream-K slots, when
// the GEMM on the copies has a stream-K part, follow the copies.
int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }
size_t round256(size_t x) { return (x + 255) / 256 * 256; }

struct StageLayout {
    bool a = false, b = false;       // which operands are copied
    size_t a_bytes = 0, b_bytes = 0; // their copies, each rounded to 256 bytes
    size_t bytes() const { return a_bytes + b_bytes; }
};

StageLayout stage_layout(bool stage_a, bool stage_b, int64_t M, int64_t N, int64_t K) {
    StageLayout L;
    L.a = stage_a;
    L.b = stage_b;
    L.a_bytes = stage_a ? round256((size_t)M * (size_t)round8(K) * 2) : 0;
    L.b_bytes = stage_b ? round256((size_t)K * (size_t)round8(N) * 2) : 0;
    return L;
}

// Workspace bytes of the stream-K part of a GEMM of these sizes on the TMA
// path (0: none).
size_t tma_streamk_bytes(int64_t M, int64_t N, int64_t K, int sms) {
    const SkPlan plan = streamk_plan(M, N, K, 1, sms);
    return plan.dp_tiles < 0 ? 0 : streamk_bytes(plan.ctas);
}

// The staged GEMM: one copy kernel for the operands that need it, then the
// kernel the TMA path would run on aligned operands of these sizes -- the
// CTA pair or the single-CTA kernel, with the stream-K schedule when the
// workspace also has room for its slots -- storing C by TMA when its rows
// allow, else with predicated stores.  The GEMM is a programmatic dependent
// of the copy, so its set-up overlaps the copy.
int launch_staged(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                  const StageLayout &L, void *workspace, size_t workspace_bytes,
                  cudaStream_t stream, DeviceState *ds) {
    namespace G = gemmrelu::stage;
    char *ws = static_cast<char *>(workspace);
    const uint16_t *a = static_cast<const uint16_t *>(A), *b = static_cast<const uint16_t *>(B);
    int64_t lda = K, ldb = N;
    G::Params sp{};
    int jobs = 0;
    int64_t chunks[2] = {0, 0};
    if (L.a) {
        lda = round8(K);
        sp.job[jobs] = G::Job{a, reinterpret_cast<uint16_t *>(ws), M, K, lda};
        chunks[jobs++] = M * (lda / 8);
        a = reinterpret_cast<const uint16_t *>(ws);
    }
    if (L.b) {
        ldb = round8(N);
        sp.job[jobs] = G::Job{b, reinterpret_cast<uint16_t *>(ws + L.a_bytes), K, N, ldb};
        chunks[jobs++] = K * (ldb / 8);
        b = reinterpret_cast<const uint16_t *>(ws + L.a_bytes);
    }
    sp.chunks0 = chunks[0];
    sp.total = chunks[0] + chunks[1];
    if (jobs == 1)
        sp.job[1] = sp.job[0];   // (never read: every chunk index is below chunks0)
    if (jobs > 0) {              // (none when only C's rows are unaligned)
        const int64_t blocks = std::max<int64_t>(
            1, std::min<int64_t>((sp.total + 255) / 256, (int64_t)8 * ds->sms));
        const int rc =
            launch_kernel(G::stage_rows_kernel, (unsigned)blocks, 256, 0, stream, false, 1, sp);
        if (rc != GEMMRELU_OK)
            return rc;
    }
    const SkPlan plan = streamk_plan(M, N, K, 1, ds->sms);
    StreamK sk;
    if (plan.dp_tiles >= 0 && workspace_bytes >= L.bytes() + streamk_bytes(plan.ctas)) {
        char *skw = ws + L.bytes();
        sk.dp_tiles = plan.dp_tiles;
        sk.ctas = plan.ctas;
        sk.part = reinterpret_cast<float *>(skw);
        sk.head = reinterpret_cast<float *>(skw + (size_t)plan.ctas * kSkSlotBytes);
        sk.flags = reinterpret_cast<uint32_t *>(skw + 2 * (size_t)plan.ctas * kSkSlotBytes);
        sk.epoch = next_epoch();
    }
    // (streamk_plan chose between the two kernels by the same use_pair)
    if (use_pair(M, N, ds->sms, 1))
        return launch_pair(a, b, C, M, N, K, stream, ds, sk, lda, ldb);
    return launch_single_cta(a, lda, b, ldb, C, M, N, K, true, stream, ds, sk);
}

// ---------------------------------------------------------------- split-K
namespace S = gemmrelu::splitk;

int split_bms(int64_t M) {
    if (M <= 16)
        return 16;
    if (M <= 32)
        return 32;
    if (M <= 64)
        return 64;
    return 128;
}

// k per pipeline stage of the split-K kernel instantiated for `bms`.
int64_t split_super_k(int bms) { return (int64_t)S::BK * S::kbs_for(bms); }

int64_t split_super_blocks(int64_t K, int bms) {
    return (K + split_super_k(bms) - 1) / split_super_k(bms);
}

int effective_splits(int64_t K, int bms, int split_k) {
    return (int)std::max<int64_t>(1, std::min<int64_t>(split_k, split_super_blocks(K, bms)));
}

struct SplitLayout {
    int bms, splits;
    bool cluster;  // pieces reduced inside a cluster: no workspace, one kernel
    int64_t n_tiles, m_tiles, part_bytes;
};

// The cluster form splits a tile's S pieces evenly over a CTA pair and keeps
// one TMEM accumulator per piece, double-buffered: S even and S * BMS <= 512
// TMEM columns.  It serves M <= 64; for larger M the two-stage form, whose
// units spread over every SM, measured faster.
bool split_cluster_ok(int splits, int bms) {
    return g_force_split.load() == 0 && splits >= 2 && splits % 2 == 0 && splits * bms <= 512 &&
           bms <= 64;
}

SplitLayout split_layout(int64_t M, int64_t N, int64_t K, int split_k) {
    SplitLayout L{};
    L.bms = split_bms(M);
    L.splits = effective_splits(K, L.bms, split_k);
    L.cluster = split_cluster_ok(L.splits, L.bms);
    L.n_tiles = (N + S::BNT - 1) / S::BNT;
    L.m_tiles = (M + L.bms - 1) / L.bms;
    L.part_bytes = L.cluster ? 0 : (int64_t)L.splits * M * N * 4;
    return L;
}

// Stage 2 launch: programmatic dependent of the partial kernel just queued on
// `stream`, so its CTAs can become resident while stage 1 drains.
int launch_split_reduce(const float *part, void *C, int64_t M, int64_t N, int splits,
                        cudaStream_t stream, DeviceState *ds) {
    const int64_t groups = M * (N / 4);
    const int64_t blocks = std::max<int64_t>(
        1, std::min<int64_t>((groups + 255) / 256, (int64_t)8 * ds->sms));
    const int c_vec8 = aligned(C, 8) ? 1 : 0;
    return launch_kernel(S::gemm_relu_splitk_reduce_kernel, (unsigned)blocks, 256, 0, stream, false,
                         1, part, static_cast<uint16_t *>(C), (int)M, (int)N, splits, c_vec8);
}

template <int BMS>
int launch_split_bms(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                     const SplitLayout &L, void *ws, cudaStream_t stream, DeviceState *ds,
                     int bms_index) {
    S::Params p{};
    p.part = static_cast<float *>(ws);
    p.C = static_cast<uint16_t *>(C);
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.num_sb = (int)split_super_blocks(K, BMS);
    p.splits = L.splits;
    p.n_tiles = L.n_tiles;
    p.m_tiles = L.m_tiles;
    p.split_major = kSplitMajor;
    p.drop_arrive = g_drop_arrive.load();
    p.wait_limit_ns = wait_limit_ns();
    constexpr int kSuperK = S::Cfg<BMS, false>::kSuperK;
    CUtensorMap mA, mB;
    if (!make_map(&mA, A, M, K, S::BK, BMS) || !make_map(&mB, B, K, N, 64, kSuperK))
        return GEMMRELU_ERR_LAUNCH;
    if (!L.cluster) {
        using G = S::Cfg<BMS, false>;
        p.num_units = L.n_tiles * L.m_tiles * L.splits;
        auto kern = S::gemm_relu_splitk_kernel<BMS, false>;
        if (!ensure_smem_attr(ds->attr_split[bms_index], kern, G::kSmemBytes))
            return GEMMRELU_ERR_LAUNCH;
        const int64_t grid = std::min<int64_t>(p.num_units, ds->sms);
        const int rc = launch_kernel(kern, (unsigned)grid, 192, G::kSmemBytes, stream, false, 1,
                                     mA, mB, p);
        if (rc != GEMMRELU_OK)
            return rc;
        return launch_split_reduce(p.part, C, M, N, L.splits, stream, ds);
    }
    // cluster form: persistent CTA pairs, one tile at a time each
    using G = S::Cfg<BMS, true>;
    p.num_units = L.n_tiles * L.m_tiles;
    auto kern = S::gemm_relu_splitk_kernel<BMS, true>;
    if (!ensure_smem_attr(ds->attr_split_cluster[bms_index], kern, G::kSmemBytes))
        return GEMMRELU_ERR_LAUNCH;
    int &resident = ds->split_pairs[bms_index];
    if (resident <= 0) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)(2 * std::max(1, ds->sms / 2)));
        cfg.blockDim = dim3(192);
        cfg.dynamicSmemBytes = G::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            return GEMMRELU_ERR_LAUNCH;
        }
        resident = n;
    }
    const int64_t pairs = std::min<int64_t>(p.num_units, resident);
    return launch_kernel(kern, (unsigned)(2 * pairs), 192, G::kSmemBytes, stream, false, 2, mA, mB,
                         p);
}

// ---------------------------------------------------------------- skinny shapes
// A plain launch of a skinny shape (M <= 64) whose 128 x 256 tiles would keep
// fewer than half of the SMs busy runs as a split of K in two, in the
// CTA-pair form: two CTAs per 128-column tile, each streaming half of K, the
// halves added in a fixed order on chip -- one kernel, no workspace.
bool use_skinny_split(const void *A, const void *B, int64_t M, int64_t N, int64_t K, int sms) {
    if (g_force_kernel.load() != 0 || g_force_split.load() != 0 || M > 64)
        return false;
    if (!tma_ok(A, K) || !tma_ok(B, N))
        return false;
    const int64_t tiles = ((M + 127) / 128) * ((N + 255) / 256);
    if (2 * tiles > sms)
        return false;
    const SplitLayout L = split_layout(M, N, K, 2);
    return L.splits == 2 && L.cluster;
}

int launch_skinny_split(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream, DeviceState *ds) {
    const SplitLayout L = split_layout(M, N, K, 2);
    switch (L.bms) {
    case 16:
        return launch_split_bms<16>(A, B, C, M, N, K, L, nullptr, stream, ds, 0);
    case 32:
        return launch_split_bms<32>(A, B, C, M, N, K, L, nullptr, stream, ds, 1);
    default:
        return launch_split_bms<64>(A, B, C, M, N, K, L, nullptr, stream, ds, 2);
    }
}

// ---------------------------------------------------------------- attention forward
namespace FA = gemmrelu::attn;

// [batch][seq][heads][d] fp16 as a 4-D tensor (d innermost), boxes of 64 d x
// 1 head x 128 rows x 1 batch, 128-byte swizzle, zero fill outside.
bool make_bshd_map(CUtensorMap *map, const void *ptr, int64_t batch, int64_t seq, int64_t heads,
                   int64_t d) {
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)seq, (cuuint64_t)batch};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)(heads * d) * 2,
                             (cuuint64_t)(seq * heads * d) * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)FA::BM, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD>
int launch_attention(const CUtensorMap &mQ, const CUtensorMap &mK, const CUtensorMap &mV,
                     const FA::Params &p, cudaStream_t stream, bool &attr_done) {
    using G = FA::Cfg<HD>;
    auto kern = FA::flash_attention_fwd_kernel<HD>;
    if (!ensure_smem_attr(attr_done, kern, G::kSmemBytes))
        return GEMMRELU_ERR_LAUNCH;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)p.ctas_x, (unsigned)p.heads, (unsigned)p.batch);
    cfg.blockDim = dim3(FA::kThreads);
    cfg.dynamicSmemBytes = G::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = GEMMRELU_PDL ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_status(cudaLaunchKernelEx(&cfg, kern, mQ, mK, mV, p));
}

// ---------------------------------------------------------------- no-alloc scratch
// Split-K scratch for gemm_relu_f16_splitk_noalloc: a fixed array in every
// device's copy of this module, so callers that cannot allocate still get a
// workspace.  Host code must not use the symbol's host-side name as a device
// address; it looks the address up once per device instead.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMMRELU_NOALLOC_SCRATCH_BYTES];

void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call per device, with that device current).
int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return GEMMRELU_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return GEMMRELU_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GEMMRELU_OK;
}

// gemm_relu_f16_splitk and gemm_relu_f16_splitk_noalloc: one routing
// decision and one layout per call.  With `noalloc`, the partials of the
// two-stage form go to g_noalloc_scratch instead of a caller workspace; the
// other forms need no scratch, so only the two-stage form is held to the
// array's size.
int splitk_run(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int split_k,
               void *workspace, size_t workspace_bytes, bool noalloc, cudaStream_t s) {
    int rc = check_args(A, B, C, M, N, K);
    if (rc != GEMMRELU_OK)
        return rc;
    if (split_k < 1)
        return GEMMRELU_ERR_WORKSPACE;
    if (M == 0 || N == 0)
        return GEMMRELU_OK;
    DeviceState *ds = nullptr;
    rc = current_device_state(&ds);
    if (rc != GEMMRELU_OK)
        return rc;
    if (K == 0)
        return zero_fill(C, M, N, s);
    const SplitLayout L = split_layout(M, N, K, split_k);
    if (L.splits <= 1 || !tma_ok(A, K) || !tma_ok(B, N))
        return launch_fused(A, B, C, M, N, K, s, ds);
    const size_t need = (size_t)L.part_bytes;
    if (noalloc && need > 0) {
        if (need > GEMMRELU_NOALLOC_SCRATCH_BYTES)
            return GEMMRELU_ERR_SCRATCH_LIMIT;
        rc = noalloc_scratch(&workspace);
        if (rc != GEMMRELU_OK)
            return rc;
        workspace_bytes = GEMMRELU_NOALLOC_SCRATCH_BYTES;
    }
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return GEMMRELU_ERR_WORKSPACE;
    switch (L.bms) {
    case 16:
        return launch_split_bms<16>(A, B, C, M, N, K, L, workspace, s, ds, 0);
    case 32:
        return launch_split_bms<32>(A, B, C, M, N, K, L, workspace, s, ds, 1);
    case 64:
        return launch_split_bms<64>(A, B, C, M, N, K, L, workspace, s, ds, 2);
    default:
        return launch_split_bms<128>(A, B, C, M, N, K, L, workspace, s, ds, 3);
    }
}

}  // namespace

// ==================================================================== C ABI
extern "C" {

int gemm_relu_f16(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                  void *stream) {
    int rc = check_args(A, B, C, M, N, K);
    if (rc != GEMMRELU_OK)
        return rc;
    if (M == 0 || N == 0)
        return GEMMRELU_OK;
    DeviceState *ds = nullptr;
    rc = current_device_state(&ds);
    if (rc != GEMMRELU_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return zero_fill(C, M, N, s);
    return launch_fused(A, B, C, M, N, K, s, ds);
}

size_t gemm_relu_f16_streamk_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return 0;
    DeviceState *ds = nullptr;
    if (current_device_state(&ds) != GEMMRELU_OK)
        return 0;
    // rows TMA cannot describe: room for both copies before the stream-K slots
    const size_t copies = (K % 8 != 0 || N % 8 != 0) ? stage_layout(true, true, M, N, K).bytes() : 0;
    return copies + tma_streamk_bytes(M, N, K, ds->sms);
}

int gemm_relu_f16_streamk(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                          void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_args(A, B, C, M, N, K);
    if (rc != GEMMRELU_OK)
        return rc;
    if (M == 0 || N == 0)
        return GEMMRELU_OK;
    DeviceState *ds = nullptr;
    rc = current_device_state(&ds);
    if (rc != GEMMRELU_OK)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return zero_fill(C, M, N, s);
    const int path = fused_path(A, B, C, M, N, K);
    if (path == 2) {
        // Copy the operands TMA cannot describe into the workspace, then the
        // TMA kernel; without room for the copies (only possible when the
        // pitches are aligned and a base is not), the predicated-load kernel.
        // Odd pitches: the workspace must be what the query reports (room
        // for both copies and the stream-K slots), whichever operands this
        // call's pointers need.
        const StageLayout L = stage_layout(!tma_ok(A, K), !tma_ok(B, N), M, N, K);
        const bool odd = K % 8 != 0 || N % 8 != 0;
        const size_t need = odd ? stage_layout(true, true, M, N, K).bytes() +
                                      tma_streamk_bytes(M, N, K, ds->sms)
                                : L.bytes();
        const bool room = need == 0 ||
                          (workspace && workspace_bytes >= need && aligned(workspace, 16));
        if (room)
            return launch_staged(A, B, C, M, N, K, L, workspace, workspace ? workspace_bytes : 0, s,
                                 ds);
        if (odd)
            return GEMMRELU_ERR_WORKSPACE;
        return launch_fused(A, B, C, M, N, K, s, ds);
    }
    const SkPlan plan = streamk_plan(M, N, K, path, ds->sms);
    if (plan.dp_tiles < 0)
        return launch_fused(A, B, C, M, N, K, s, ds);
    if (!workspace || workspace_bytes < streamk_bytes(plan.ctas) || !aligned(workspace, 16))
        return GEMMRELU_ERR_WORKSPACE;
    StreamK sk;
    sk.dp_tiles = plan.dp_tiles;
    char *ws = static_cast<char *>(workspace);
    sk.part = reinterpret_cast<float *>(ws);
    sk.head = reinterpret_cast<float *>(ws + (size_t)plan.ctas * kSkSlotBytes);
    sk.flags = reinterpret_cast<uint32_t *>(ws + 2 * (size_t)plan.ctas * kSkSlotBytes);
    sk.epoch = next_epoch();
    sk.ctas = plan.ctas;
    if (plan.pair)
        return launch_pair(A, B, C, M, N, K, s, ds, sk);
    return launch_fused(A, B, C, M, N, K, s, ds, sk);
}

size_t gemm_relu_f16_splitk_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k) {
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || split_k < 1)
        return 0;
    const SplitLayout L = split_layout(M, N, K, split_k);
    if (L.splits <= 1)
        return 0;
    return (size_t)L.part_bytes;
}

int gemm_relu_f16_splitk(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                         int split_k, void *workspace, size_t workspace_bytes, void *stream) {
    return splitk_run(A, B, C, M, N, K, split_k, workspace, workspace_bytes, false,
                      static_cast<cudaStream_t>(stream));
}

int gemm_relu_f16_splitk_noalloc(const void *A, const void *B, void *C, int64_t M, int64_t N,
                                 int64_t K, int split_k, void *stream) {
    return splitk_run(A, B, C, M, N, K, split_k, nullptr, 0, true,
                      static_cast<cudaStream_t>(stream));
}

int flash_attention_f16(const void *Q, const void *K, const void *V, void *O, int64_t batch,
                        int64_t seq, int64_t heads, int64_t head_dim, int causal, void *stream) {
    if (batch < 0 || seq < 0 || heads < 0 || batch > 65535 || heads > 65535 || seq > kMaxDim ||
        (head_dim != 64 && head_dim != 128))
        return GEMMRELU_ERR_INVALID_ARG;
    if (batch == 0 || seq == 0 || heads == 0)
        return GEMMRELU_OK;
    // batch * heads * head_dim <= 65535^2 * 128 < 2^39 fits; the element
    // count is bounded by 2^40 without forming the product with seq
    const int64_t bhd = batch * heads * head_dim;
    if (!Q || !K || !V || !O || !aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) ||
        !aligned(O, 16) || seq > ((int64_t)1 << 40) / bhd)
        return GEMMRELU_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    int rc = current_device_state(&ds);
    if (rc != GEMMRELU_OK)
        return rc;
    CUtensorMap mQ, mK, mV;
    if (!make_bshd_map(&mQ, Q, batch, seq, heads, head_dim) ||
        !make_bshd_map(&mK, K, batch, seq, heads, head_dim) ||
        !make_bshd_map(&mV, V, batch, seq, heads, head_dim))
        return GEMMRELU_ERR_LAUNCH;
    FA::Params p{};
    p.O = static_cast<uint16_t *>(O);
    p.batch = (int)batch;
    p.seq = (int)seq;
    p.heads = (int)heads;
    p.q_tiles = (int)((seq + FA::BM - 1) / FA::BM);
    p.ctas_x = (p.q_tiles + FA::kTiles - 1) / FA::kTiles;
    p.causal = causal ? 1 : 0;
    p.scale = (float)(1.4426950408889634 / std::sqrt((double)head_dim));  // log2(e) / sqrt(d)
    p.drop_arrive = g_drop_arrive.load();
    p.wait_limit_ns = wait_limit_ns();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (head_dim == 64)
        return launch_attention<64>(mQ, mK, mV, p, s, ds->attr_attn[0]);
    return launch_attention<128>(mQ, mK, mV, p, s, ds->attr_attn[1]);
}

int gemm_relu_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMMRELU_ERR_CUDA;
    unsigned int st = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&st, gemmrelu::g_status, sizeof(st)) != cudaSuccess)
        return GEMMRELU_ERR_CUDA;
    if (st != 0 && cudaMemcpyToSymbol(gemmrelu::g_status, &zero, sizeof(zero)) != cudaSuccess)
        return GEMMRELU_ERR_CUDA;
    return (int)st;
}

const char *gemm_relu_strerror(int code) {
    switch (code) {
    case GEMMRELU_OK: return "ok";
    case GEMMRELU_ERR_INVALID_ARG: return "invalid argument";
    case GEMMRELU_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case GEMMRELU_ERR_WORKSPACE: return "split_k < 1 or workspace missing, misaligned or too small";
    case GEMMRELU_ERR_LAUNCH: return "CUDA error configuring or launching a kernel";
    case GEMMRELU_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case GEMMRELU_ERR_CUDA: return "CUDA runtime error";
    case GEMMRELU_ERR_SCRATCH_LIMIT:
        return "split-K scratch needed exceeds the built-in GEMMRELU_NOALLOC_SCRATCH_BYTES buffer";
    default: return "unknown status";
    }
}

int gemm_relu_f16_path(const void *A, const void *B, const void *C, int64_t M, int64_t N,
                       int64_t K) {
    return fused_path(A, B, C, M, N, K);
}

int gemm_relu_f16_kernel(const void *A, const void *B, const void *C, int64_t M, int64_t N,
                         int64_t K) {
    const int path = fused_path(A, B, C, M, N, K);
    if (path <= 0)
        return path;
    DeviceState *ds = nullptr;
    if (current_device_state(&ds) != GEMMRELU_OK)
        return -2;
    return kernel_for(A, B, C, M, N, K, ds->sms);
}

int gemm_relu_tile_coord(int64_t tile, int64_t m_tiles, int64_t n_tiles, int panel, int64_t *m_blk,
                         int64_t *n_blk) {
    if (!m_blk || !n_blk || m_tiles <= 0 || n_tiles <= 0 || panel <= 0 || tile < 0 ||
        tile >= m_tiles * n_tiles)
        return -1;
    int64_t mb, nb;
    tile_coord(tile, m_tiles, n_tiles, panel, mb, nb);
    *m_blk = mb;
    *n_blk = nb;
    return 0;
}

int gemm_relu_debug_force_kernel(int which) {
    if (which < 0 || which > 4)
        return GEMMRELU_ERR_INVALID_ARG;
    g_force_kernel.store(which);
    return GEMMRELU_OK;
}

int gemm_relu_debug_force_split(int which) {
    if (which < 0 || which > 1)
        return GEMMRELU_ERR_INVALID_ARG;
    g_force_split.store(which);
    return GEMMRELU_OK;
}

int gemm_relu_debug_streamk(int mode) {
    if (mode < 0 || mode > 3)
        return GEMMRELU_ERR_INVALID_ARG;
    g_sk_mode.store(mode);
    return GEMMRELU_OK;
}

int gemm_relu_debug_streamk_plan(int64_t M, int64_t N, int64_t K, int path, int sms,
                                 int64_t *dp_tiles, int64_t *ctas, int *pair) {
    if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || sms < 2 ||
        (path != 1 && path != 2) || !dp_tiles || !ctas || !pair)
        return GEMMRELU_ERR_INVALID_ARG;
    const SkPlan plan = streamk_plan(M, N, K, path, sms);
    *dp_tiles = plan.dp_tiles;
    *ctas = plan.dp_tiles < 0 ? 0 : plan.ctas;
    *pair = plan.pair ? 1 : 0;
    return GEMMRELU_OK;
}

int gemm_relu_debug_streamk_pieces(int pieces) {
    if (pieces != 0 && (pieces < 2 || pieces > 8))
        return GEMMRELU_ERR_INVALID_ARG;
    g_sk_pieces.store(pieces);
    return GEMMRELU_OK;
}

int gemm_relu_debug_set_panel(int rows) {
    if (rows < 0 || rows % 128 != 0)
        return GEMMRELU_ERR_INVALID_ARG;
    g_panel_rows.store(rows);
    return GEMMRELU_OK;
}

int gemm_relu_debug_set(int drop_arrive, int64_t wait_limit_ns_arg) {
    g_drop_arrive.store(drop_arrive ? 1 : 0);
    g_wait_limit_ns.store(wait_limit_ns_arg > 0 ? wait_limit_ns_arg : 0);
    return GEMMRELU_OK;
}

}  // extern "C"
