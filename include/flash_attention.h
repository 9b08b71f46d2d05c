/*
 * flash_attention.h -- attention forward on GB300 (sm_103a), C ABI of
 * libgemmrelu.so (the same library as gemm_relu.h; status codes, the device
 * watchdog and gemm_relu_status / gemm_relu_strerror are shared).
 */
#ifndef FLASH_ATTENTION_H
#define FLASH_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#include "gemm_relu.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * flash_attention_f16 -- O = softmax(Q K^T / sqrt(d)) V for every batch and
 * head, the FlashAttention forward of the TileLang tutorial pages (section
 * "FlashAttention": online softmax over blocks of keys, base-2 exponentials
 * with log2(e) / sqrt(d) folded in, fp32 accumulation, P rounded to fp16 for
 * the second product, causal mode cut at the diagonal).
 *
 * Q, K, V, O : DEVICE pointers to fp16 arrays of shape [batch][seq][heads][d]
 *              (row-major; the pages' "bshd"), 16-byte aligned, on the
 *              current CUDA device; the caller owns them.  O must not overlap
 *              Q, K or V (not checked).
 * batch, seq, heads >= 0 (0 in any of them: nothing to do, returns OK);
 *              batch and heads at most 65535.
 * head_dim   : 64 or 128 (else GEMMRELU_ERR_INVALID_ARG).
 * causal     : nonzero -> query i attends to keys 0..i only.
 * stream     : cudaStream_t to launch on (NULL = legacy default stream).
 *
 * One CTA per 128-row query tile of one (batch, head): TMA loads of Q and of
 * 128-key blocks of K and V, tcgen05.mma for S = Q K^T and O += P V with both
 * accumulators in TMEM, one thread per query row for the softmax.  The
 * summation order is fixed: the same call gives the same bits.
 *
 * Returns GEMMRELU_OK or an error code; asynchronous on `stream`.  Device-side
 * timeouts surface through gemm_relu_status.
 */
int flash_attention_f16(const void *Q, const void *K, const void *V, void *O,
                        int64_t batch, int64_t seq, int64_t heads, int64_t head_dim,
                        int causal, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FLASH_ATTENTION_H */
