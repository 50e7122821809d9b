/*
 * bi_attention.h — C ABI of the batch-invariant decode attention (in libbi_gemm.so), sm_103a.
 *
 * For each query token t — request b = q_seq[t] at position p = q_pos[t] — and each query head
 * h (KV head h / G, G = num_q_heads / num_kv_heads):
 *
 *     o[t, h, :] = sum_{j <= p} softmax_j(scale * q[t, h, :] . K_b[j, h/G, :]) V_b[j, h/G, :]
 *
 * the causal attention of the nondeterminism article ("Batch-invariant attention"), over a paged
 * KV cache that already holds positions 0..p of every request (the article's fix for the
 * cache-boundary problem: the cache and page table are updated before the attention kernel, so
 * the layout seen by the kernel does not depend on how many tokens a step processes).
 * K_b[j, kh, :] = k_cache[page_table[b][j / page_size], j % page_size, kh, :] (V alike).
 *
 * Batch invariance: the article's split-KV with a FIXED SPLIT SIZE (not a fixed split count):
 * the keys 0..p are cut at multiples of `split_size` positions, split s always covers
 * [s * split_size, min((s + 1) * split_size, p + 1)), every split is reduced in one fixed order
 * (the same block size, staging and thread mapping for every split), and the n splits are
 * merged in one fixed order: four consecutive groups of ceil(n / 4) splits, each summed in
 * ascending s, the group sums added in order (n is a function of p alone).  Nothing depends on
 * the number of query tokens, on the other requests, on the
 * request's index b, on where its pages sit, or on whether its earlier tokens were processed in
 * the same call (chunked prefill): o[t] is a function of q[t], p and K_b, V_b[0..p] only, bit for
 * bit.  Arithmetic: scores on the tensor cores (bf16 products, fp32 accumulation, one fixed
 * instruction shape) times scale * log2(e); weights exp2 of the score minus the split's maximum
 * in fp32; the weighted sum of the values on the tensor cores with each weight split into two
 * bf16 parts (16 significant bits) and fp32 accumulation in ascending position; fp32 merge and
 * division; one bf16 rounding at the end.
 *
 * Conventions (as in bi_gemm.h, whose BI_GEMM_* return codes these functions use):
 *   - q [T, num_q_heads, head_dim] and o likewise, bf16 row-major; k_cache, v_cache
 *     [num_pages, page_size, num_kv_heads, head_dim] bf16; page_table int32 [num_seqs,
 *     max_pages] (entry -1 = no page); q_seq, q_pos int32 [T].  All DEVICE pointers owned by the
 *     caller; q, o, k_cache, v_cache 16-byte aligned, the int32 arrays 4-byte aligned (else
 *     BI_GEMM_ERR_ALIGNMENT).
 *   - Inputs the host cannot see (a q_seq outside [0, num_seqs), a negative q_pos, a position
 *     whose page-table entry lies past max_pages or names no page in [0, num_pages), a q_pos
 *     above max_pos) are caught by the kernels: the token's output is then undefined and
 *     bi_attention_get_device_error reports BI_GEMM_ERR_INVALID_ARG.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  A handle is
 *     not thread-safe and must not be used on two streams at once.
 */
#ifndef BI_ATTENTION_H
#define BI_ATTENTION_H

#include <stdint.h>

#include "bi_gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bi_attention* bi_attention_t;

typedef struct {
  int32_t num_q_heads, num_kv_heads, head_dim, page_size;
  int32_t split_size;       /* positions per split (fixed for the handle)                      */
  int32_t threads;          /* threads per block of the attention kernel                      */
  int32_t stage_positions;  /* positions staged in shared memory at a time                    */
  int32_t max_ctas;         /* persistent grid bound: resident blocks per SM x SMs            */
  int32_t num_sms;
  int32_t tma_pages;        /* 1: pages are loaded as TMA boxes by a producer warp (page sizes
                               8, 16, 32, 64); 0: rows are copied by every thread (cp.async)  */
  int32_t ring_stages;      /* depth of the staging ring                                       */
} bi_attention_config;

/* Create a handle.  Requirements (else BI_GEMM_ERR_UNSUPPORTED): head_dim 64 or 128;
 * num_q_heads / num_kv_heads = G in {1, 2, 4, 8}; page_size >= 1; split_size (0 = 512) a
 * multiple of 128 up to 1024; an sm_103 device.  scale must be finite and > 0 (else
 * BI_GEMM_ERR_INVALID_ARG; 1 / sqrt(head_dim) is the usual value).  Checks on the arguments
 * come before any CUDA call.  *out is NULL on failure. */
int bi_attention_create(bi_attention_t* out, int64_t num_q_heads, int64_t num_kv_heads,
                        int64_t head_dim, int64_t page_size, float scale, int64_t split_size);

/* o = attention(q) for T query tokens.  max_pos: an upper bound (on the host) of every q_pos;
 * it sizes the workspace and the grid and changes no result.  T = 0 queues nothing.  The run
 * grows the handle's workspace (stream-ordered cudaMallocAsync) when T or max_pos outgrow it
 * (BI_GEMM_ERR_OOM if that fails), then queues three kernels on `stream`: a plan of the
 * (token, KV head, split) units, the attention of every unit, and the merge of the splits of
 * tokens that have more than one.  Asynchronous.
 *
 * Two attention kernels, with the same arithmetic and the same bits: for page sizes 8, 16, 32
 * and 64 (a 64-position stage is whole pages) a producer warp loads every page's rows of a KV
 * head as 3-D TMA boxes into a ring that runs ahead across units, and four warps compute (three
 * blocks per SM with a deeper ring, or, for a call that fits one round of four blocks per SM but
 * not of three, four blocks with a shallower ring); for other page sizes (or a cache of 2^31 rows
 * or more) every thread copies 16-byte row chunks with cp.async.  The waits of the TMA kernel on its ring are bounded (2 s): past the limit the
 * block stops, its output is undefined and bi_attention_get_device_error reports
 * BI_GEMM_ERR_TIMEOUT. */
int bi_attention_run(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                     const int32_t* q_pos, const void* k_cache, const void* v_cache,
                     int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                     int64_t max_pages, int64_t max_pos, void* o, void* stream);

/* Workspace bytes a run with T tokens and the bound max_pos needs. */
int bi_attention_workspace_size(bi_attention_t h, int64_t T, int64_t max_pos, uint64_t* bytes);

/* Synchronise `stream`; BI_GEMM_ERR_TIMEOUT if a bounded wait expired, else
 * BI_GEMM_ERR_INVALID_ARG if a kernel caught a bad input, since the last call (the status is then
 * cleared); BI_GEMM_ERR_CUDA if synchronisation failed; else BI_GEMM_OK. */
int bi_attention_get_device_error(bi_attention_t h, void* stream);

int bi_attention_get_config(bi_attention_t h, bi_attention_config* c);

/* Release the handle and its workspace (NULL is a no-op). */
int bi_attention_destroy(bi_attention_t h);

#ifdef __cplusplus
}
#endif
#endif
