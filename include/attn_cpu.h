/*
 * attn_cpu.h -- C ABI of the online-softmax attention forward on the host CPU
 * (libattn_cpu.so).
 *
 * The same operation and conventions as attn_fwd in attn.h (layout [B, H, N, d] bf16,
 * LSE [B, H, Nq] fp32, key padding, bottom-right causal mask, fully masked rows O = 0 and
 * LSE = -inf), computed on the CPU with the recurrence of "FlashAttention math"
 * (aicassindra.com), section "The block-wise update, and the full algorithm", blocked the
 * way its section "Why the same math matters on a CPU" describes: a tile of 64 query rows
 * stays in cache while blocks of 64 keys and values stream through once, so the N x N
 * score matrix is never formed.  Arithmetic is fp32 (scores, running max, denominator
 * and accumulator), the output is rounded to bf16 once.
 *
 * This is a separate library for hosts without a GPU or for CPU-side work; the GPU
 * entry points never call it and it never calls them.
 */
#ifndef ATTN_CPU_H_
#define ATTN_CPU_H_

#include <stdint.h>

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_fwd_cpu -- attention forward on host memory.
 *   Q, K, V, O  host bf16 codes (uint16) [B, H, Nq | Nk, d], contiguous; O is written.
 *   LSE         host fp32 [B, H, Nq], written.
 *   d           1 .. 256.  scale finite and > 0.  causal, key_padding_lens (host int32[B]
 *               or NULL): as attn_fwd.
 *   num_threads worker threads (0: one per online CPU).
 * Synchronous.  Returns ATTN_OK, ATTN_ERR_NULLPTR, ATTN_ERR_BAD_SHAPE,
 * ATTN_ERR_UNSUPPORTED_D, ATTN_ERR_BAD_ARG or ATTN_ERR_LAUNCH (a thread failed to start;
 * the call then finishes on the threads it has).
 */
attn_status attn_fwd_cpu(const uint16_t* Q, const uint16_t* K, const uint16_t* V, uint16_t* O, float* LSE, int B,
                         int H, int Nq, int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                         int num_threads);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_CPU_H_ */
