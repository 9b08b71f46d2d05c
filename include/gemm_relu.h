/*
 * gemm_relu.h -- C ABI of libgemmrelu.so: fused fp16 GEMM + ReLU on GB300 (sm_103a).
 *
 *     C = fp16( max( A . B , 0 ) )
 *
 * A is M x K, B is K x N, C is M x N; all three are dense, row-major fp16
 * (leading dimensions K, N and N).  Products accumulate in fp32 inside the
 * tensor cores; ReLU is applied to the fp32 accumulator and the result is
 * rounded to fp16 (round-to-nearest-even) once, on the way out.
 *
 * The operation is the one defined by the FP16 GEMM + ReLU quickstart of
 * "TileLang 编程基本知识点" (section 二: fp16 operands, fp32 accumulator
 * fragment, element-wise max(x, 0) epilogue, lowering to fp16 on the store)
 * and by "在 TileLang 中編寫高效能核心：從 GEMM 到 MLA" (section "編寫一個
 * GEMM": C = ReLU(A @ B) with the ReLU fused before the write-back).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers A, B, C and `workspace` are DEVICE pointers on the current CUDA
 *    device; the caller allocates and owns them.  The library allocates no
 *    memory per call.  Per device it keeps a status word and the fixed
 *    scratch array of gemm_relu_f16_splitk_noalloc in static device variables.
 *  - Pointers must be at least 2-byte aligned.  When A, B and C are 16-byte
 *    aligned and K and N are multiples of 8 (16-byte row pitches), operands
 *    move by TMA; otherwise by plain predicated loads and stores.  Both give
 *    the same result.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous on it.  The return code covers argument checks and launch
 *    errors; a device-side watchdog timeout is reported by gemm_relu_status().
 *  - M, N, K must lie in [0, 2^31 - 1].  M == 0 or N == 0: nothing is written,
 *    GEMMRELU_OK.  K == 0: C is filled with +0 (the empty sum, then ReLU).
 *  - C must not overlap A, B or the workspace (not checked).
 *  - Errors leave C unspecified.  No entry point aborts the process.
 */
#ifndef GEMM_RELU_H
#define GEMM_RELU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMMRELU_OK = 0,
    GEMMRELU_ERR_INVALID_ARG = 1,        /* null pointer with non-empty size, negative or too large dims, misaligned pointer */
    GEMMRELU_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute capability 10.3 */
    GEMMRELU_ERR_WORKSPACE = 3,          /* split_k < 1, or workspace null / smaller than the query */
    GEMMRELU_ERR_LAUNCH = 4,             /* CUDA reported an error configuring or launching a kernel */
    GEMMRELU_ERR_TIMEOUT = 5,            /* a bounded device-side wait expired (from gemm_relu_status) */
    GEMMRELU_ERR_CUDA = 6,               /* another CUDA runtime error (e.g. while reading the status) */
    GEMMRELU_ERR_SCRATCH_LIMIT = 7       /* gemm_relu_f16_splitk_noalloc: problem needs more scratch
                                            than GEMMRELU_NOALLOC_SCRATCH_BYTES */
} gemmrelu_status;

/*
 * gemm_relu_f16 -- C = fp16(max(A . B, 0)).
 *
 * One fused kernel, chosen per shape:
 *   - M >= 256 and N >= 256 with TMA-capable A, B, C: 256 x 256 tiles on CTA
 *     pairs (tcgen05.mma.cta_group::2), when that needs no more waves than
 *     one CTA per 128 x 256 tile and the 128 x 128 tiles outnumber the SMs;
 *   - M <= 2, or M <= 4 unless the case below applies with one CTA pair
 *     per 128 columns all resident at once (2 * ceil(N / 128) <= SMs), with
 *     TMA-capable A and B: the GEMV kernel -- B streamed through shared
 *     memory, fp32 multiply-adds on the CUDA cores, K chunks reduced in a
 *     fixed order inside a thread-block cluster (the GEMV pattern of
 *     "TileLang CUDA 核心编程模式" section 4);
 *   - M <= 64 with TMA-capable A and B whose 128 x 256 tiles would keep
 *     fewer than half of the SMs busy: gemm_relu_f16_splitk's CTA-pair form
 *     with split_k = 2 (one kernel, no workspace; identical bits to that
 *     call);
 *   - otherwise one CTA per 128 x 256 (or 128 x 128) tile: TMA (or predicated
 *     loads) into a multistage shared-memory ring, tcgen05.mma into a TMEM
 *     fp32 accumulator, ReLU + fp16 cast in the epilogue, TMA (or
 *     predicated) stores; persistent grid, grouped (L2-friendly) tile order.
 * Every choice sums in a fixed order: the same call gives the same bits.
 *
 * Returns GEMMRELU_OK or an error code; asynchronous on `stream`.
 */
int gemm_relu_f16(const void *A, const void *B, void *C,
                  int64_t M, int64_t N, int64_t K, void *stream);

/*
 * gemm_relu_f16_streamk_workspace_bytes -- bytes of device workspace that
 * gemm_relu_f16_streamk needs for these sizes on the current device (its SM
 * count decides the schedule): the stream-K schedule's slots (none when the
 * call would run no stream-K part) and, when K or N is not a multiple of 8,
 * room for aligned copies of A and B before them.  0 for invalid arguments,
 * or when no CUDA device is available.
 */
size_t gemm_relu_f16_streamk_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * gemm_relu_f16_streamk -- C = fp16(max(A . B, 0)) like gemm_relu_f16, with a
 * stream-K schedule for the tiles of a partial wave, and operands whose rows
 * TMA cannot describe copied once into aligned rows of the workspace.
 *
 * "TileLang tutorial" (chapter "Persistent kernel") names the problem: when
 * the number of output tiles is not a multiple of the number of SMs, the
 * last wave runs on part of the GPU only; stream-K splits the remaining work
 * over all CTAs along K.  Here all full waves but the last run data-parallel
 * (one 128 x 256 tile per CTA, or a 256 x 256 tile per CTA pair, at a time);
 * the k blocks of the remaining tiles are divided into one equal contiguous
 * range per worker.  That applies only when the plain schedule's partial last
 * wave would idle long enough to pay for the cut tiles' fix-up: (ceil(W) - W)
 * times the k blocks of a tile at least 40, for W = tiles / workers.  With
 * fewer single-CTA tiles than SMs and a long K (M > 64), each tile's k blocks
 * are cut into k blocks / 128 + 1 equal pieces (2 to 8, pieces x tiles <= SMs)
 * when that shortens the work of a CTA by at least 32 k blocks and the
 * operand several tiles share fits in half of L2.  A tile cut between workers is
 * summed in fp32 before the ReLU and the fp16 store: each cut is settled by
 * whichever of its two sides gets there second, each side publishing its
 * fp32 part through `workspace` unless the other's is already there, and no
 * CTA ever waits for another, so the kernel needs no guarantee that its CTAs
 * run at the same time.  A tile cut more than once is summed from its last
 * k blocks backwards, p0 + (p1 + (p2 + ...)) over its pieces in k order,
 * whatever the order of arrival (fp32 addition is commutative), so the
 * result is the same from run to run.
 *
 * Operands: when A's or B's rows do not start on 16-byte boundaries (a row
 * pitch that is not a multiple of 8 elements, or an unaligned base), the
 * call first copies that operand into rows of pitch round_up(cols, 8) in
 * the workspace (one extra kernel), then runs on the copies the kernel the
 * TMA path would choose for these sizes (CTA pairs or single CTAs, with the
 * stream-K schedule above when it applies); when C's rows are unaligned, that
 * kernel stores C with predicated stores.  Where the copies run on the
 * single-CTA kernel with no tile cut, the result has the same bits as
 * gemm_relu_f16's predicated-load kernel.
 *
 * workspace: device buffer of at least
 *            gemm_relu_f16_streamk_workspace_bytes(M, N, K) bytes, 16-byte
 *            aligned; its contents need no initialisation.  Calls that may
 *            run concurrently on the GPU must use distinct workspaces.
 *            Returns GEMMRELU_ERR_WORKSPACE when it is needed and missing,
 *            smaller than that or misaligned.  With aligned pitches but an
 *            unaligned base, the copies are made when the workspace has room
 *            for them, else gemm_relu_f16's predicated-load kernel runs.
 * When no stream-K schedule applies and the operands' rows are aligned, the
 * call runs gemm_relu_f16's kernel and leaves the workspace untouched.
 */
int gemm_relu_f16_streamk(const void *A, const void *B, void *C,
                          int64_t M, int64_t N, int64_t K,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * gemm_relu_f16_splitk_workspace_bytes -- bytes of device workspace that
 * gemm_relu_f16_splitk needs for these sizes (0 if no workspace is needed).
 * Host-only; never touches the device.  Returns 0 for invalid arguments.
 */
size_t gemm_relu_f16_splitk_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

/*
 * gemm_relu_f16_splitk -- the same C = fp16(max(A . B, 0)), with the K range
 * cut into `split_k` contiguous pieces computed by different CTAs.
 *
 * Follows the split-K scheme of "TileLang 编程基本知识点" section 5.1 (work
 * split over K pieces, each piece offsetting only K) with that page's advice
 * for reproducible results: instead of fp32 atomic adds into C, every piece's
 * raw fp32 partial (no ReLU) is kept and the partials are summed in the fixed
 * order 0..split_k-1 before the ReLU and the fp16 cast.  Results are
 * bit-identical from run to run, and the same in both forms below:
 *   - M <= 64 and clamped split_k even, with split_k * R <= 512 (R = 16, 32
 *     or 64 for M <= 16, <= 32, <= 64): one kernel.  A CTA pair (a
 *     thread-block cluster of 2) computes the split_k pieces of a tile, half
 *     each, and continues the ordered sum from one CTA to the other through
 *     distributed shared memory; no workspace is used (the workspace query
 *     returns 0).
 *   - any other clamped split_k: two stages on `stream`.  Stage 1 writes the
 *     partials to `workspace`; stage 2, a programmatic dependent launch of
 *     stage 1, sums them, applies ReLU and writes C.
 *
 * The product is computed as C^T = B^T . A^T so that small M maps onto the
 * narrow (N) side of the MMA; this suits skinny, memory-bound shapes.
 *
 * split_k  : >= 1.  K is processed in stages of 64, 128 or 256 k (256 when
 *            M <= 32); split_k is clamped to the number of such stages.
 * workspace: device buffer of at least
 *            gemm_relu_f16_splitk_workspace_bytes(M, N, K, split_k) bytes
 *            (split_k * M * N fp32 partials in the two-stage form), 16-byte
 *            aligned; may be NULL when that query returns 0.  Its contents
 *            need no initialisation; calls that may run concurrently on the
 *            GPU must use distinct workspaces.
 * Needs A, B 16-byte aligned with K and N multiples of 8 (TMA operands);
 * otherwise, or when the clamped split_k is 1, the call runs gemm_relu_f16's
 * kernel and leaves the workspace untouched.
 */
int gemm_relu_f16_splitk(const void *A, const void *B, void *C,
                         int64_t M, int64_t N, int64_t K, int split_k,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * gemm_relu_f16_splitk_noalloc -- gemm_relu_f16_splitk for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry point.
 *
 * Who needs it: code that may not call cudaMalloc or any allocator -- for
 * example a host framework that owns every byte of device memory through its
 * own pool and forbids libraries to allocate behind its back, a serving loop
 * that bans allocation after warm-up so its latency and footprint stay
 * fixed, or a plugin that is handed only input and output pointers and has
 * no way to obtain a workspace.  Such callers pass A, B and C exactly as for
 * gemm_relu_f16_splitk; the split-K partial sums live in a fixed scratch
 * array compiled into this library instead of a caller workspace.  Nothing
 * is allocated by this call.
 *
 * Scratch: GEMMRELU_NOALLOC_SCRATCH_BYTES (8 MiB) of device memory in a
 * static device array.  Every GPU that loads the library holds it until the
 * process exits.  Only the two-stage form of gemm_relu_f16_splitk uses it:
 * a call that runs that form needs
 * gemm_relu_f16_splitk_workspace_bytes(M, N, K, split_k) bytes of it, and
 * if that is more than the array holds the call returns
 * GEMMRELU_ERR_SCRATCH_LIMIT and launches nothing.  Calls that run the
 * CTA-pair form or fall back to the unsplit kernel (split_k clamped to 1, or
 * operands that cannot use TMA) need no scratch and run whatever the
 * workspace query says.  (16 x 8192 x 8192 at split_k 8 takes the CTA-pair
 * form; forced into the two-stage form it needs 4 MiB.)
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  Make that first call
 * before any stream capture begins.  A failed look-up returns
 * GEMMRELU_ERR_CUDA.
 *
 * Sharing: every call on a device uses the same array, and it keeps whatever
 * the previous call left there.  Every byte a call reads from it is first
 * written by the same call, so leftover contents are harmless and nothing
 * needs clearing between calls.  Calls whose kernels may overlap on the GPU
 * (for example on two streams without ordering between them) race on the
 * array and give undefined results: order them on one stream or with events.
 *
 * Everything else -- arguments, layouts, alignment, the choice of form, the
 * fallback to the unsplit kernel, status reporting -- is as for
 * gemm_relu_f16_splitk, and so are the result's bits.  The test hooks below
 * must not change while a call is being made.
 */
#define GEMMRELU_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int gemm_relu_f16_splitk_noalloc(const void *A, const void *B, void *C,
                                 int64_t M, int64_t N, int64_t K, int split_k, void *stream);

/*
 * gemm_relu_status -- synchronise `stream`, then return and clear the current
 * device's watchdog word: GEMMRELU_OK, or GEMMRELU_ERR_TIMEOUT if a bounded
 * wait inside a kernel expired since the last call (that kernel's output is
 * then unspecified; the CUDA context stays usable).  Returns GEMMRELU_ERR_CUDA
 * if the synchronisation or the read fails.
 */
int gemm_relu_status(void *stream);

/* gemm_relu_strerror -- static, human-readable text for a status code. */
const char *gemm_relu_strerror(int code);

/*
 * gemm_relu_f16_path -- which operand path gemm_relu_f16 would take for these
 * arguments: 1 = TMA loads and stores, 2 = predicated loads and stores,
 * 0 = nothing to launch (empty output or K == 0), -1 = invalid arguments.
 * Host-only; never touches the device.
 */
int gemm_relu_f16_path(const void *A, const void *B, const void *C,
                       int64_t M, int64_t N, int64_t K);

/* The kernels gemm_relu_f16 chooses from (see gemm_relu_f16_kernel). */
typedef enum {
    GEMMRELU_KERNEL_PAIR = 1,        /* 256 x 256 tiles on CTA pairs (tcgen05 cta_group::2) */
    GEMMRELU_KERNEL_ONE_CTA_256 = 2, /* 128 x 256 tiles, one CTA each */
    GEMMRELU_KERNEL_ONE_CTA_128 = 3, /* 128 x 128 tiles, one CTA each */
    GEMMRELU_KERNEL_PREDICATED = 4,  /* predicated loads and stores, 128 x 128 tiles */
    GEMMRELU_KERNEL_GEMV = 5,        /* CUDA-core GEMV for decode-like rows */
    GEMMRELU_KERNEL_SPLITK_PAIR = 6  /* split-K CTA-pair form with split_k = 2 */
} gemmrelu_kernel;

/*
 * gemm_relu_f16_kernel -- which kernel gemm_relu_f16 would launch for these
 * arguments on the current device (the choice depends on its SM count and on
 * the gemm_relu_debug_force_* hooks): a gemmrelu_kernel code, 0 = nothing to
 * launch (empty output or K == 0), -1 = invalid arguments, -2 = no usable
 * CUDA device.  Launches nothing.
 */
int gemm_relu_f16_kernel(const void *A, const void *B, const void *C,
                         int64_t M, int64_t N, int64_t K);

/*
 * gemm_relu_tile_coord -- the tile rasteriser, evaluated on the host (the
 * kernels run the same function on the device).  Maps linear tile id `tile`
 * in [0, m_tiles * n_tiles) to (m_blk, n_blk): tiles are taken in panels of
 * `panel` consecutive M blocks; inside a panel the id walks down the column
 * (M fastest) before moving to the next N block -- the grouped launch order
 * that "在 TileLang 中編寫高效能核心" (section "編寫一個 GEMM",
 * T.use_swizzle(panel_size=4, order="col")) uses for L2 reuse.
 * Returns 0, or -1 for out-of-range arguments.
 */
int gemm_relu_tile_coord(int64_t tile, int64_t m_tiles, int64_t n_tiles, int panel,
                         int64_t *m_blk, int64_t *n_blk);

/*
 * gemm_relu_debug_set -- test hook.  drop_arrive != 0 makes the next launches
 * skip one producer arrival in CTA 0 (so the consumer's bounded wait expires
 * and gemm_relu_status reports GEMMRELU_ERR_TIMEOUT); wait_limit_ns sets the
 * bound of every device-side wait (<= 0 restores the default of one second).
 * Affects the calling process only.  Returns GEMMRELU_OK.
 */
int gemm_relu_debug_set(int drop_arrive, int64_t wait_limit_ns);

/*
 * gemm_relu_debug_force_kernel -- test hook.  Selects the kernel that
 * gemm_relu_f16 (and the unsplit fallbacks of the other entry points) runs:
 * 0 = automatic choice (default), 1 = one CTA per 128 x 256 tile, 2 = one CTA
 * per 128 x 128 tile, 3 = CTA pairs on 256 x 256 tiles (TMA operands only;
 * others take the one-CTA kernel), 4 = the GEMV kernel where it applies
 * (M <= 8, TMA-capable A and B; else the automatic choice).  All give
 * results within the same tolerance.  Affects the calling process only.  Returns GEMMRELU_OK, or
 * GEMMRELU_ERR_INVALID_ARG for another value.
 */
int gemm_relu_debug_force_kernel(int which);

/*
 * gemm_relu_debug_force_split -- test hook.  0 = gemm_relu_f16_splitk picks
 * its form as documented there (default); 1 = always the two-stage form (the
 * workspace query follows the setting).  Both forms give identical bits.
 * Affects the calling process only.  Returns GEMMRELU_OK, or
 * GEMMRELU_ERR_INVALID_ARG for another value.
 */
int gemm_relu_debug_force_split(int which);

/*
 * gemm_relu_debug_set_panel -- test hook.  Sets the height of the tile
 * rasteriser's panels (see gemm_relu_tile_coord) in output rows: a multiple
 * of 128, or 0 for the library's own choice (default).  Every panel height
 * gives the same results; it changes only the order in which tiles are
 * computed, and so L2 reuse.  Affects the calling process only.  Returns
 * GEMMRELU_OK, or GEMMRELU_ERR_INVALID_ARG for another value.
 */
int gemm_relu_debug_set_panel(int rows);

/*
 * gemm_relu_debug_streamk -- test hook for the stream-K fix-up of a tile cut
 * between two workers.  0 (default): the side that holds the k blocks left
 * of the cut adds the other side's published piece when it is already there.
 * 1: that side always publishes its own piece first, so the second side to
 * arrive finishes the cut from global memory.  2: as 1, and the side right of
 * the cut also waits about 0.2 ms before publishing.  3: as 1, and the side
 * left of the cut waits about 0.2 ms instead.  Modes 2 and 3 exercise the
 * two orders of arrival (and, for a tile cut more than once, which worker
 * carries the sum on to the next cut).  All modes give the same bits.
 * Affects the calling process only.  Returns GEMMRELU_OK, or
 * GEMMRELU_ERR_INVALID_ARG for another value.
 */
int gemm_relu_debug_streamk(int mode);

/*
 * gemm_relu_debug_streamk_pieces -- test hook.  The number of pieces each
 * tile's k blocks are cut into by gemm_relu_f16_streamk's sub-wave schedule
 * (fewer single-CTA tiles than SMs): 2 .. 8, or 0 for the library's choice
 * (default: k blocks / 128 + 1, from 2 to 8).  With 2 each tile is cut once
 * in the middle; with 3 or more, tiles have middle pieces and are settled
 * through chains of cuts.  Affects the
 * calling process only.  Returns GEMMRELU_OK, or GEMMRELU_ERR_INVALID_ARG
 * for another value.
 */
int gemm_relu_debug_streamk_pieces(int pieces);

/*
 * gemm_relu_debug_streamk_plan -- the stream-K schedule gemm_relu_f16_streamk
 * would use for these sizes on operands of path `path` (1 = TMA-capable rows,
 * 2 = rows TMA cannot describe; the staged path plans its copies as path 1)
 * on a GPU of `sms` SMs: *dp_tiles = the data-parallel tiles before the
 * stream-K part, or -1 for no stream-K part; *ctas = the grid of the
 * stream-K launch (0 when none); *pair = 1 for the CTA-pair kernel.  Honours
 * the gemm_relu_debug_force_kernel and gemm_relu_debug_streamk_pieces hooks.
 * Host-only; never touches the device.  Returns GEMMRELU_OK, or
 * GEMMRELU_ERR_INVALID_ARG for invalid sizes, path, sms < 2 or null outputs.
 */
int gemm_relu_debug_streamk_plan(int64_t M, int64_t N, int64_t K, int path, int sms,
                                 int64_t *dp_tiles, int64_t *ctas, int *pair);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_RELU_H */
