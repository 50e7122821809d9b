/*
 * bi_gemm_controls.h — TEST-ONLY C ABI of libbi_gemm_controls.so (kept beside the tests, outside
 * the product's include/).
 *
 * Deliberately batch-variant negative controls, for proving that the batch-invariance
 * harness can fail, and a failure-injection hook for the bounded in-kernel waits.  The
 * product library (bi_gemm.h) never contains or calls any of this.  Handles created here
 * belong to this library only; do not pass them to libbi_gemm.so or vice versa.
 *
 * The two defects are those of "[BI][DSv4] Make mHC tilelang ops batch invariant"
 * (github.com/aoshen02/vllm/pull/22, "What"): a K-split count derived from the token count,
 * n_sms // cdiv(num_tokens, 64), and a second implementation used at num_tokens <= 16.
 * Argument rules, layouts, ownership and return codes are those of bi_gemm.h.
 */
#ifndef BI_GEMM_CONTROLS_H
#define BI_GEMM_CONTROLS_H

#include <stdint.h>

#include "../../include/bi_attention.h"
#include "../../include/bi_gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* bi_gemm_create_ex with split_k (0 = automatic) and timeout_ns (0 = default). */
int bi_ctl_create(bi_gemm_t* out, int64_t K, int64_t N, int dtype, int scale_layout,
                  int32_t split_k, uint64_t timeout_ns);
int bi_ctl_destroy(bi_gemm_t h);
int bi_ctl_get_device_error(bi_gemm_t h, void* stream);

/* The batch-invariant product path as compiled into this library. */
int bi_ctl_run(bi_gemm_t h, const void* x, int64_t M, const void* W,
               const bi_gemm_scales* scales, void* y, void* stream);

/* Control N1: the split count used for M rows, n_sms / cdiv(M, 64) clamped to [1, KB]. */
int bi_ctl_msplit_count(bi_gemm_t h, int64_t M);

/* Control N1: run with that M-dependent split count (fixed-order merge, but the K ranges
 * and hence the reduction tree change with M). */
int bi_ctl_run_msplit(bi_gemm_t h, const void* x, int64_t M, const void* W,
                      const bi_gemm_scales* scales, void* y, void* stream);

/* Control N2: M <= 16 runs a CUDA-core fp32 FMA kernel (ascending k), larger M the product
 * kernel.  bf16 inputs only (BI_GEMM_ERR_UNSUPPORTED for MXFP8). */
int bi_ctl_run_smallm_fork(bi_gemm_t h, const void* x, int64_t M, const void* W, void* y,
                           void* stream);

/* Failure injection: the TMA producer withholds the first stage of each CTA's first tile,
 * so the MMA issuer's bounded wait expires.  The kernel records an error in the status word
 * (read by bi_ctl_get_device_error as BI_GEMM_ERR_TIMEOUT), lets in-flight copies finish,
 * frees its tensor memory and returns; y is undefined.  No GPU fault is raised. */
int bi_ctl_run_stall(bi_gemm_t h, const void* x, int64_t M, const void* W,
                     const bi_gemm_scales* scales, void* y, void* stream);

/* Failure injection for the shared split-K merge (used when every split unit has its own
 * resident CTA and a sub-tile's partials exceed 24 KB): split 0 of every tile never counts
 * its arrival, so the other split CTAs' bounded waits for it expire.  The status word then reads
 * BI_GEMM_ERR_TIMEOUT; y is undefined; the next run resets the arrival counters. */
int bi_ctl_run_skip_arrival(bi_gemm_t h, const void* x, int64_t M, const void* W,
                            const bi_gemm_scales* scales, void* y, void* stream);

/* Control N3 (RMSNorm of bf16 rows, include/bi_rmsnorm.h, written in fp32 before the bf16
 * rounding so that any change in the reduction order shows).  mkeyed = 0: the product's threads
 * per row, fixed from d (must be batch-invariant).  mkeyed = 1: threads per row chosen from the
 * batch size, 1024 while M <= 16 and the product's count above (must not be).  x, g bf16 and y
 * fp32 [M, d] device pointers, 16-byte aligned; codes as bi_rmsnorm_run. */
int bi_ctl_rmsnorm_f32(const void* x, int64_t M, int64_t d, const void* g, float eps, void* y,
                       int32_t mkeyed, void* stream);

/* This library's own copies of bi_attention_create / _run / _get_device_error / _destroy
 * (include/bi_attention.h, same arguments and codes): a handle made here is used only with
 * this library's functions. */
int bi_ctl_attention_create(bi_attention_t* out, int64_t num_q_heads, int64_t num_kv_heads,
                            int64_t head_dim, int64_t page_size, float scale, int64_t split_size);
int bi_ctl_attention_run(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                         const int32_t* q_pos, const void* k_cache, const void* v_cache,
                         int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                         int64_t max_pages, int64_t max_pos, void* o, void* stream);
int bi_ctl_attention_get_device_error(bi_attention_t h, void* stream);
int bi_ctl_attention_destroy(bi_attention_t h);

/* Failure injection for the TMA page-box attention kernel (include/bi_attention.h; a handle
 * whose config has tma_pages = 1, else BI_GEMM_ERR_UNSUPPORTED): bi_attention_run with block 0's
 * producer never issuing its first load and the ring waits limited to timeout_ns (> 0).  Block
 * 0's consumer waits expire, the block stops and waits (bounded) for its copies in flight;
 * bi_attention_get_device_error then reads BI_GEMM_ERR_TIMEOUT and o is undefined.  The handle
 * stays usable. */
int bi_ctl_attention_stall(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                           const int32_t* q_pos, const void* k_cache, const void* v_cache,
                           int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                           int64_t max_pages, int64_t max_pos, void* o, uint64_t timeout_ns,
                           void* stream);

/* bi_attention_run with the kernel pinned (kernel = 1: the TMA page-box kernel, for a handle
 * whose config has tma_pages = 1, else BI_GEMM_ERR_UNSUPPORTED; kernel = 2: the row-copy
 * kernel), so that tests can run both kernels on the same calls whichever the product picks. */
int bi_ctl_attention_run_kernel(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                                const int32_t* q_pos, const void* k_cache, const void* v_cache,
                                int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                                int64_t max_pages, int64_t max_pos, void* o, int32_t kernel, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* BI_GEMM_CONTROLS_H */
