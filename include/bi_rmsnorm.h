/*
 * bi_rmsnorm.h — C ABI of the batch-invariant RMSNorm (in libbi_gemm.so), sm_103a (GB300).
 *
 *     y[i, j] = bf16( (x[i, j] * r_i) * g[j] ),   r_i = 1 / sqrt( (sum_j x[i, j]^2) / d + eps )
 *
 * The definition is the one of the nondeterminism article ("Batch-invariant RMSNorm":
 * RMSNorm(x_i) = x_i / sqrt(mean_j x_ij^2 + eps) * gamma, evaluated as
 * x * rsqrt(mean(x ** 2)) * weight), with fp32 arithmetic and one round-to-nearest-even to
 * bf16 at the end.  Batch invariance: the article's data-parallel strategy, one row's whole
 * reduction inside one thread block, with a reduction tree fixed at bi_rmsnorm_create from d
 * alone — each of `threads` threads sums the squares of its own elements in ascending order
 * (fused multiply-add), the 32 lanes of a warp combine by a fixed xor butterfly, and the warp
 * partials are added in warp order.  Neither M nor the block that processes a row changes
 * any of it, so output row i depends only on x[i], g and eps, bit for bit, for every M.
 *
 * Conventions (as in bi_gemm.h, whose BI_GEMM_* return codes these functions use):
 *   - Return value BI_GEMM_OK (0) or a negative BI_GEMM_ERR_* code; nothing aborts or prints.
 *   - Layouts: x[M, d], y[M, d] row-major bf16 (d contiguous), g[d] bf16.  No strides.
 *   - x, g, y are DEVICE pointers owned by the caller, on the device that was current at
 *     bi_rmsnorm_create, each 16-byte aligned (else BI_GEMM_ERR_ALIGNMENT).  y may be x
 *     itself (in place: every row is read whole before it is written); any other overlap of
 *     y with x or g is undefined.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream); the run is
 *     asynchronous on it.  A handle is not thread-safe.
 *   - Rows whose sum of squares overflows fp32 (|x| around 2^63 / sqrt(d) and above) give
 *     zeros or NaN, as an fp32 evaluation of the definition does.
 */
#ifndef BI_RMSNORM_H
#define BI_RMSNORM_H

#include <stdint.h>

#include "bi_gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bi_rmsnorm* bi_rmsnorm_t;

/* The fixed configuration of a handle (chosen from d and the SM count, never from M). */
typedef struct {
  int32_t d;                   /* row length                                                 */
  int32_t threads;             /* threads per row (one thread block), multiple of 32, 128..1024 */
  int32_t vectors_per_thread;  /* 16-byte vectors (8 elements) per thread: thread t owns
                                  vectors t, t + threads, ... of the row                      */
  int32_t max_ctas;            /* grid bound of the persistent launch: resident blocks per
                                  SM x SMs (a block loops over rows blockIdx.x, blockIdx.x +
                                  gridDim.x, ..., loading its next row while it reduces one).
                                  A batch with more rows than this, but few enough for every
                                  row to get a resident block of its own when the registers
                                  are capped at half, runs that capped launch instead, one
                                  block per row; the arithmetic is the same.                   */
  int32_t num_sms;
} bi_rmsnorm_config;

/* Create a handle for rows of length d with the given eps (added in fp32).
 * Requirements: 8 <= d <= 32768 and d % 8 == 0 (16-byte rows), else BI_GEMM_ERR_UNSUPPORTED;
 * eps finite and >= 0 and out != NULL, else BI_GEMM_ERR_INVALID_ARG (both checked before any
 * CUDA call); a device that is not sm_103 gives BI_GEMM_ERR_UNSUPPORTED; a failing CUDA
 * query BI_GEMM_ERR_CUDA; out of host memory BI_GEMM_ERR_OOM.  *out is NULL on failure. */
int bi_rmsnorm_create(bi_rmsnorm_t* out, int64_t d, float eps);

/* y = RMSNorm(x) * g for M rows.  M = 0 queues nothing and returns BI_GEMM_OK; M < 0 or a
 * null handle or pointer gives BI_GEMM_ERR_INVALID_ARG (also when the current device is not
 * the handle's); a misaligned pointer BI_GEMM_ERR_ALIGNMENT; a failed launch
 * BI_GEMM_ERR_CUDA.  Allocates nothing; safe inside CUDA graph capture. */
int bi_rmsnorm_run(bi_rmsnorm_t h, const void* x, int64_t M, const void* g, void* y, void* stream);

/* Copy the handle's configuration into *c (BI_GEMM_ERR_INVALID_ARG on null arguments). */
int bi_rmsnorm_get_config(bi_rmsnorm_t h, bi_rmsnorm_config* c);

/* Release the handle (NULL is a no-op returning BI_GEMM_OK). */
int bi_rmsnorm_destroy(bi_rmsnorm_t h);

#ifdef __cplusplus
}
#endif
#endif
