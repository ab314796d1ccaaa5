/*
 * lm_head.h -- C ABI of the bf16 vocabulary projection (lm_head) of a
 * decode/verify step: logits[m][v] = sum_h x[m][h] * W[v][h] for M <= 16
 * tokens, fp32 logits, bf16 inputs.
 *
 * Source (page title and section): "How Ling-3.0-flash reduces batch 1
 * decoding latency by 54% on 4 Blackwell GPUs", section "bf16 router gate and
 * lm_head": at batch 1 the lm_head is pure bandwidth -- every decode step
 * cold-reads the whole (vocab-parallel) projection and no arithmetic hides
 * the read; keeping the weight in bf16 instead of fp32 halves those bytes.
 * The post's model has hidden 2560 and a vocabulary of about 157k tokens.
 *
 * One persistent kernel per call (one CTA per SM) streams the weight once,
 * chained to the previous work on the stream with Programmatic Dependent
 * Launch and capturable in a CUDA graph.  Conventions (bf16, device/host
 * pointers, status codes, moe_last_error(), one handle per host thread and
 * stream, sm_103a only) are those of moe.h.
 */
#ifndef WSE_LM_HEAD_H
#define WSE_LM_HEAD_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_lm_head moe_lm_head_t; /* opaque; owned by the library */

#define MOE_LM_HEAD_MAX_TOKENS 16

/*
 * moe_lm_head_create -- copy and re-lay out the projection weight.
 *   hidden   256, 512, 1024, 1280, 2048, 2560, 3072 or 4096 (the kernel
 *            instances).
 *   vocab    1..16,777,216 rows (any count: the last tile is zero-padded).
 *   w        device bf16 [vocab][hidden] row-major, 16-byte aligned; read
 *            once here, not kept (the caller may free it afterwards).
 * Synchronises the device before it reads w (work still writing w on any
 * stream finishes first).  Returns NULL on error (moe_last_error() says
 * why): bad sizes or pointers, a device other than sm_103a, out of memory.
 */
moe_lm_head_t* moe_lm_head_create(int hidden, int vocab, const void* w);

/*
 * moe_lm_head_forward -- logits of M tokens.
 *   x        device bf16 [M][hidden], 16-byte aligned.
 *   logits   device fp32 [M][vocab], 4-byte aligned; fully overwritten.
 *   M        0 <= M <= 16 (0: no work, MOE_OK).
 *   stream   CUDA stream; the call is asynchronous (no host synchronisation,
 *            no allocation) and PDL-chained to the previous work on it.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG (null/misaligned pointers),
 * MOE_ERR_UNSUPPORTED (M > 16) or MOE_ERR_CUDA (launch failure).  Device-side
 * trouble (a bounded wait that ran out) is reported by
 * moe_lm_head_get_status, never by a trap.
 */
int moe_lm_head_forward(moe_lm_head_t* h, const void* x, float* logits, int M, moe_stream_t stream);

/* Sticky device status word of the handle (synchronises the device): 0 or
 * MOE_ERR_DEVICE_TIMEOUT, with moe_last_error() naming the wait. */
int moe_lm_head_get_status(moe_lm_head_t* h);

/* Frees the handle (NULL-safe); synchronises the device first. */
void moe_lm_head_destroy(moe_lm_head_t* h);

#ifdef __cplusplus
}
#endif

#endif /* WSE_LM_HEAD_H */
