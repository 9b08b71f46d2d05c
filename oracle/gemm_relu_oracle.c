/*
 * CPU oracle for the fused GEMM + ReLU:  C = fp16( max( A . B , 0 ) ).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file.  Its users are the tests, the smoke check of the package
 * entry point and the CPU-baseline leg of the benchmark.  It shares no code,
 * header, table or helper with the CUDA library: it is written directly from
 * the definition of the operation on the pages, slow and obviously correct.
 *
 * What it follows:
 *   - "TileLang 编程基本知识点" (ggaaooppeenngg blog), section 二, the FP16 GEMM +
 *     ReLU quickstart: A is M x K and B is K x N, both fp16 and row-major; the
 *     product accumulates into a wider (fp32) accumulator, the epilogue takes
 *     max(x, 0) on the accumulator, and only then is the value lowered to fp16.
 *   - "在 TileLang 中編寫高效能核心：從 GEMM 到 MLA" (atlascloud), section
 *     "編寫一個 GEMM": the same C = ReLU(A @ B) with the ReLU applied to the
 *     accumulator fragment before the write-back.
 *   - "TileLang 编程基本知识点", section 六 ①: check against a reference that
 *     accumulates in higher precision than the kernel, not against fp16 a@b.
 *
 * Readings taken where the pages are silent:
 *   - The accumulator here is fp64, which is stronger than the pages' fp32:
 *     every fp16 x fp16 product is exact in fp64 (11 + 11 significand bits),
 *     and the K-term fp64 sum is within ~K * 2^-53 relative of exact.
 *   - "Lowered to fp16" is read as IEEE-754 binary16 round-to-nearest,
 *     ties-to-even, with magnitudes that round above 65504 becoming infinity.
 *     The rounding below is written from the binary16 format definition.
 *   - ReLU maps every non-positive sum (including -0) to +0.
 *   - K = 0 gives the empty sum 0, hence C = 0.
 *
 * Build:  gcc -O2 -ffp-contract=off -shared -fPIC  (see oracle/build_oracle.py)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* ---- binary16 <-> double ------------------------------------------------ */

/* Decode an IEEE-754 binary16 bit pattern to double (exact).
 * Layout: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.        */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f + 1024), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even.
 *
 * For |x| in binade e (2^e <= |x| < 2^(e+1)), e >= -14, the binary16 spacing
 * is 2^(e-10); below 2^-14 the spacing stays 2^-24 (subnormals).  Scaling |x|
 * by 2^(10-e) puts the representable neighbours on consecutive integers, so
 * the rounding is an integer round-half-even of the scaled value.  With the
 * scaled integer m, the bit pattern is ((e + 14) << 10) + m: this covers the
 * subnormals (e = -14, m < 1024), the normals (m in [1024, 2048)) and the
 * carry into the next binade (m == 2048) in one expression.               */
uint16_t oracle_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7e00u);
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0)
        return sign;
    if (a >= 65536.0)                       /* beyond every finite binary16 */
        return (uint16_t)(sign | 0x7c00u);

    int ex;
    (void)frexp(a, &ex);                    /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                         /* 2^e <= a < 2^(e+1)          */
    if (e < -14)
        e = -14;
    double scaled = ldexp(a, 10 - e);       /* exact: power-of-two scale   */
    double fl = floor(scaled);
    double rem = scaled - fl;               /* exact                        */
    uint32_t m = (uint32_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (m & 1u)))
        m += 1u;
    uint32_t bits = ((uint32_t)(e + 14) << 10) + m;
    if (bits >= 0x7c00u)
        bits = 0x7c00u;                     /* rounds past 65504: infinity */
    return (uint16_t)(sign | bits);
}

/* ---- the operation ------------------------------------------------------- */

/* Pre-activation P[i,j] = sum_k A[i,k] * B[k,j] in fp64, k in increasing
 * order.  A: M x K row-major fp16 bits; B: K x N row-major; P: M x N.      */
void oracle_gemm_f64(const uint16_t *A, const uint16_t *B, double *P,
                     int64_t M, int64_t N, int64_t K)
{
    for (int64_t i = 0; i < M; ++i) {
        double *prow = P + i * N;
        for (int64_t j = 0; j < N; ++j)
            prow[j] = 0.0;
        /* i-k-j order: streams rows of B; each P[i,j] still sums k = 0..K-1 */
        for (int64_t k = 0; k < K; ++k) {
            double a = oracle_f16_to_f64(A[i * K + k]);
            const uint16_t *brow = B + k * N;
            for (int64_t j = 0; j < N; ++j)
                prow[j] += a * oracle_f16_to_f64(brow[j]);
        }
    }
}

/* ReLU on the accumulator, then the single rounding to fp16. */
static uint16_t relu_to_f16(double s)
{
    return oracle_f64_to_f16(s > 0.0 ? s : 0.0);
}

/* C = fp16_RNE(max(A . B, 0)) for rows [row0, row0 + nrows) of the output.
 * C points at the first of those rows (nrows x N).                         */
void oracle_gemm_relu_f16_rows(const uint16_t *A, const uint16_t *B, uint16_t *C,
                               int64_t N, int64_t K, int64_t row0, int64_t nrows)
{
    double *acc = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!acc)
        abort();
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = row0 + r;
        oracle_gemm_f64(A + i * K, B, acc, 1, N, K);
        for (int64_t j = 0; j < N; ++j)
            C[r * N + j] = relu_to_f16(acc[j]);
    }
    free(acc);
}

/* Full output, M x N. */
void oracle_gemm_relu_f16(const uint16_t *A, const uint16_t *B, uint16_t *C,
                          int64_t M, int64_t N, int64_t K)
{
    oracle_gemm_relu_f16_rows(A, B, C, N, K, 0, M);
}

/* Individual outputs C[I[t], J[t]], t < n, one dot product each (for sampled
 * checks of shapes too large for the full triple loop).                    */
void oracle_gemm_relu_f16_at(const uint16_t *A, const uint16_t *B,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t *I, const int64_t *J, int64_t n,
                             uint16_t *out)
{
    (void)M;
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = I[t], j = J[t];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += oracle_f16_to_f64(A[i * K + k]) * oracle_f16_to_f64(B[k * N + j]);
        out[t] = relu_to_f16(s);
    }
}
