/*
 * CPU oracle for attention forward:  O = fp16( softmax( Q K^T / sqrt(d) ) V ).
 *
 * TEST INFRASTRUCTURE ONLY, like gemm_relu_oracle.c (whose binary16 routines
 * it uses): nothing on the product path may include, link or call it, and it
 * shares nothing with the CUDA library.
 *
 * What it follows: the FlashAttention section of the TileLang tutorial pages
 * ("FlashAttention": problem, online softmax, kernel structure).  The kernel
 * there never forms the seq x seq score matrix and streams K/V blocks with an
 * online softmax (running row maximum, running denominator, rescaled
 * unnormalised output, base-2 exponentials with the 1/sqrt(d) folded into the
 * exponent).  All of that is a way of computing, up to rounding, the plain
 * definition written out here for each batch b, head h and query row i:
 *
 *     s_j = (sum_c Q[b,i,h,c] K[b,j,h,c]) / sqrt(d)      for visible keys j
 *     w_j = exp(s_j - max_j s_j)
 *     O[b,i,h,c] = fp16( sum_j w_j V[b,j,h,c] / sum_j w_j )
 *
 * in fp64 (every fp16 x fp16 product is exact in fp64).  The maximum is
 * subtracted only to keep exp() in range; it cancels in the ratio.
 *
 * Layout (the pages' "bshd"): Q, K, V, O are [batch][seq][heads][dim] fp16,
 * row-major.  Causal mode: key j is visible to query i iff j <= i (the pages
 * set the strictly upper triangle of the diagonal block to -inf and skip the
 * blocks past the diagonal).  Reading where the pages are silent: the output
 * is rounded once to binary16, round-to-nearest-even (oracle_f64_to_f16).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

double oracle_f16_to_f64(uint16_t h);
uint16_t oracle_f64_to_f16(double x);

/* Rows [row0, row0 + nrows) of O for one (batch b, head h). */
void oracle_attention_f16_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                               uint16_t *O, int64_t seq, int64_t heads, int64_t dim,
                               int causal, int64_t b, int64_t h, int64_t row0, int64_t nrows)
{
    const int64_t row_stride = heads * dim;                 /* elements between seq rows */
    const int64_t base = b * seq * row_stride + h * dim;    /* element (b, 0, h, 0) */
    const double inv_sqrt_d = 1.0 / sqrt((double)dim);
    double *s = (double *)malloc((size_t)(seq > 0 ? seq : 1) * sizeof(double));
    double *o = (double *)malloc((size_t)(dim > 0 ? dim : 1) * sizeof(double));
    for (int64_t i = row0; i < row0 + nrows; ++i) {
        const uint16_t *q = Q + base + i * row_stride;
        const int64_t nvis = causal ? i + 1 : seq;          /* keys 0 .. nvis-1 */
        double smax = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) {
            const uint16_t *k = K + base + j * row_stride;
            double dot = 0.0;
            for (int64_t c = 0; c < dim; ++c)
                dot += oracle_f16_to_f64(q[c]) * oracle_f16_to_f64(k[c]);
            s[j] = dot * inv_sqrt_d;
            if (s[j] > smax)
                smax = s[j];
        }
        double z = 0.0;
        for (int64_t c = 0; c < dim; ++c)
            o[c] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            const double w = exp(s[j] - smax);
            const uint16_t *v = V + base + j * row_stride;
            z += w;
            for (int64_t c = 0; c < dim; ++c)
                o[c] += w * oracle_f16_to_f64(v[c]);
        }
        uint16_t *out = O + base + i * row_stride;
        for (int64_t c = 0; c < dim; ++c)
            out[c] = oracle_f64_to_f16(o[c] / z);
    }
    free(s);
    free(o);
}

/* All of O. */
void oracle_attention_f16(const uint16_t *Q, const uint16_t *K, const uint16_t *V, uint16_t *O,
                          int64_t batch, int64_t seq, int64_t heads, int64_t dim, int causal)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t h = 0; h < heads; ++h)
            oracle_attention_f16_rows(Q, K, V, O, seq, heads, dim, causal, b, h, 0, seq);
}
