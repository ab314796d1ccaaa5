/*
 * gemv.h -- C ABI of one expert contraction on either engine of the SM:
 * y[m][r] = sum_k W[r][k] * x[m][k] for M <= 16 tokens, bf16 inputs, fp32
 * outputs, computed on the CUDA cores (fp32 FMA) or on the tensor cores
 * (mma.sync m16n8k16, bf16 in, fp32 accumulate).
 *
 * Source (page title and sections): "How Ling-3.0-flash reduces batch 1
 * decoding latency by 54% on 4 Blackwell GPUs" -- "Two kinds of idle" (a
 * small-M step is bound by the cold read of the activated expert weights)
 * and "Economics of speculation at batch 1" (verifying several tokens reads
 * the same expert weights as verifying one).  An expert that holds M_e tokens
 * does M_e / 2 multiply-adds per weight byte it streams, so at small M_e the
 * read bounds the contraction whatever does the arithmetic; these entry
 * points measure where the tensor cores start to pay (the layer kernel of
 * moe.h uses them for every group, at every M).
 *
 * The weight is streamed in the layer kernel's own layout: 8-row tiles, each
 * one contiguous block in tensor-core fragment order (moe_gemv_pack builds
 * it).  Every tile is read from HBM once for all M tokens.  Conventions
 * (status codes, moe_last_error(), device pointers, sm_103a only) are those
 * of moe.h.
 */
#ifndef WSE_GEMV_H
#define WSE_GEMV_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_GEMV_MAX_TOKENS 16
#define MOE_GEMV_MAX_K 3072

/* Engines of moe_gemv. */
#define MOE_GEMV_CUDA_CORES 0
#define MOE_GEMV_TENSOR_CORES 1

/*
 * moe_gemv_pack -- re-lay out a row-major weight for moe_gemv.
 *   w        device bf16 [rows][k] row-major, 16-byte aligned (read only).
 *   packed   device buffer of rows * k * 2 bytes, 16-byte aligned, owned by
 *            the caller; fully overwritten.
 *   rows     a positive multiple of 8; k a multiple of 32, 32..3072.
 *   stream   CUDA stream (asynchronous; no allocation).
 * Returns MOE_OK, MOE_ERR_INVALID_ARG (sizes, null or misaligned pointers)
 * or MOE_ERR_CUDA (launch failure).
 */
int moe_gemv_pack(const void* w, void* packed, int rows, int k, moe_stream_t stream);

/*
 * moe_gemv -- y = W x on the chosen engine.
 *   packed   the weight as moe_gemv_pack left it (rows x k); here k must be
 *            a multiple of 256 (the kernels stream 4 KB stages of 8 chunks).
 *   x        device bf16 [M][k] row-major, 16-byte aligned.
 *   y        device fp32 [M][rows] row-major, 4-byte aligned; fully
 *            overwritten.
 *   M        0 <= M <= 16 (0: no work, MOE_OK).
 *   engine   MOE_GEMV_CUDA_CORES or MOE_GEMV_TENSOR_CORES.
 *   stream   CUDA stream (asynchronous; no host synchronisation, no
 *            allocation; capturable in a CUDA graph).
 * Both engines sum in fp32 (in different orders, so results agree to fp32
 * rounding, not bit for bit).  Returns MOE_OK, MOE_ERR_INVALID_ARG (sizes,
 * engine, null or misaligned pointers), MOE_ERR_UNSUPPORTED (M > 16) or
 * MOE_ERR_CUDA (launch failure).
 */
int moe_gemv(const void* packed, const void* x, float* y, int rows, int k, int M, int engine,
             moe_stream_t stream);

/*
 * moe_gemv_get_status -- sticky device status of moe_gemv (synchronises the
 * device): MOE_OK, or MOE_ERR_DEVICE_TIMEOUT if a bounded wait for a staged
 * weight copy ran out (the result of that call is then undefined); reading
 * it clears it.  MOE_ERR_CUDA if the device could not be read.
 */
int moe_gemv_get_status(void);

#ifdef __cplusplus
}
#endif

#endif /* WSE_GEMV_H */
