/*
 * bi_prenorm.h — C ABI of the batch-invariant pre-norm projection of the hyper-connection (mHC)
 * block (in libbi_gemm.so), sm_103a.
 *
 *     y[i, :] = RMSNorm(x[i, :]) . W = (x[i, :] . W) / sqrt(sum_k x[i, k]^2 / K + eps)
 *
 * x[M, K] bf16 is a token's n residual streams flattened (K = n * hidden), W[K, N] bf16 the
 * projection to the mixing coefficients (N = n (n + 2): 24 for four streams), y[M, N] fp32.
 * This is the pre-norm GEMM of "[BI][DSv4] Make mHC tilelang ops batch invariant", whose
 * defect was a K-split count derived from the token count (n_sms // cdiv(num_tokens, 64)): here
 * the split is FIXED per handle, K is cut into chunks of `chunk` elements (default 512), and
 * the projection and the sum of squares of every chunk are added in ascending chunk order.  A
 * norm weight g folds into W (RMSNorm(x) * g . W = RMSNorm(x) . (diag(g) W)); this entry takes
 * the folded W.
 *
 * Arithmetic, all fixed per handle: per chunk, the projection of 16 rows on the tensor cores
 * (mma.sync m16n8k16, bf16 in, fp32 accumulate, k ascending) and each row's sum of squares in
 * fp32 (eight 64-element runs by fma, combined in a fixed order); then, per output, the chunk
 * results summed in ascending chunk order, r = correctly rounded 1/sqrt(ss / K + eps) (fp32), and
 * y = projection * r.  Row i of y depends only on x[i] and W, bit for bit, for every M.
 *
 * Conventions as in bi_gemm.h (BI_GEMM_* codes; caller-owned DEVICE pointers; x, W 16-byte
 * aligned, y 8-byte aligned, else BI_GEMM_ERR_ALIGNMENT; `stream` a cudaStream_t as void*).
 */
#ifndef BI_PRENORM_H
#define BI_PRENORM_H

#include <stdint.h>

#include "bi_gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bi_prenorm* bi_prenorm_t;

typedef struct {
  int32_t K, N;
  int32_t chunk;      /* K elements per split                         */
  int32_t splits;     /* ceil(K / chunk)                              */
  int32_t tile_rows;  /* rows of x per block (the MMA's 16)           */
} bi_prenorm_config;

/* Requirements (else BI_GEMM_ERR_UNSUPPORTED): K >= 8 and K % 8 == 0; 8 <= N <= 32 and
 * N % 8 == 0; chunk (0 = 512) a multiple of 64 up to 1024; an sm_103 device.  eps finite and
 * >= 0 (else BI_GEMM_ERR_INVALID_ARG).  Argument checks come before any CUDA call. */
int bi_prenorm_create(bi_prenorm_t* out, int64_t K, int64_t N, float eps, int64_t chunk);

/* y = RMSNorm(x) . W for M rows.  M = 0 queues nothing.  Grows the handle's workspace (the
 * per-chunk results, stream-ordered cudaMallocAsync; BI_GEMM_ERR_OOM if that fails) and queues
 * two kernels on `stream` (a block per chunk and 16-row tile; then a block per row merging
 * the chunks in order).  Asynchronous.  Calls on one handle must not overlap on the GPU. */
int bi_prenorm_run(bi_prenorm_t h, const void* x, int64_t M, const void* W, float* y, void* stream);

int bi_prenorm_get_config(bi_prenorm_t h, bi_prenorm_config* c);

/* Release the handle and its workspace (NULL is a no-op). */
int bi_prenorm_destroy(bi_prenorm_t h);

#ifdef __cplusplus
}
#endif
#endif
