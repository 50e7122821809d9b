// bi_gemm_controls.cu — TEST-ONLY library libbi_gemm_controls.so: deliberately batch-variant
// negative controls and a failure-injection hook.  Never loaded by the product path.
//
// The controls reproduce the two defects of "[BI][DSv4] Make mHC tilelang ops batch
// invariant" ("What"): a K-split count derived from the token count
// (n_sms // cdiv(num_tokens, 64)), which changes the reduction tree with the batch, and a
// second implementation for num_tokens <= 16.  The batch-invariance harness must report
// non-zero byte diffs for both, otherwise it could not tell a broken kernel from a good one
// ("Tests" on the same page: negative controls that actually fail).
//
// The product code is compiled in with its C entry points hidden, so this library's
// bi_ctl_* functions use their own copies and never mix handles with libbi_gemm.so.
#define BI_GEMM_CONTROLS 1
#define BI_GEMM_API extern "C" __attribute__((visibility("hidden")))
#include "bi_gemm.cu"
#include "bi_rmsnorm.cu"
#include "bi_attention.cu"

#include <cuda_bf16.h>

#include "../../tests/include/bi_gemm_controls.h"

#define BI_CTL_API extern "C" __attribute__((visibility("default")))

namespace {

// Second implementation for small batches: one thread per output, fp32 fused multiply-add
// in ascending k on the CUDA cores (a different rounding sequence from the tensor cores).
template <bool kOutF32>
__global__ void small_m_fma_kernel(const __nv_bfloat16* __restrict__ x,
                                   const __nv_bfloat16* __restrict__ w, void* __restrict__ y,
                                   int M, int N, int K) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  if (i >= M || j >= N) return;
  float acc = 0.f;
  for (int k = 0; k < K; ++k)
    acc = fmaf(__bfloat162float(x[(size_t)i * K + k]), __bfloat162float(w[(size_t)k * N + j]), acc);
  if (kOutF32)
    reinterpret_cast<float*>(y)[(size_t)i * N + j] = acc;
  else
    reinterpret_cast<__nv_bfloat16*>(y)[(size_t)i * N + j] = __float2bfloat16_rn(acc);
}

}  // namespace

BI_CTL_API int bi_ctl_create(bi_gemm_t* out, int64_t K, int64_t N, int dtype, int scale_layout,
                             int32_t split_k, uint64_t timeout_ns) {
  bi_gemm_options o;
  std::memset(&o, 0, sizeof(o));
  o.split_k = split_k;
  o.timeout_ns = timeout_ns;
  return bi_gemm_create_ex(out, K, N, dtype, scale_layout, &o);
}

BI_CTL_API int bi_ctl_destroy(bi_gemm_t h) { return bi_gemm_destroy(h); }

BI_CTL_API int bi_ctl_get_device_error(bi_gemm_t h, void* stream) {
  return bi_gemm_get_device_error(h, stream);
}

// The product path, as compiled into this library (reference for the controls).
BI_CTL_API int bi_ctl_run(bi_gemm_t h, const void* x, int64_t M, const void* W,
                          const bi_gemm_scales* scales, void* y, void* stream) {
  return bi_gemm_run(h, x, M, W, scales, y, stream);
}

// N1: split count = n_sms // cdiv(M, 64), clamped to [1, KB] — an M-dependent reduction tree.
BI_CTL_API int bi_ctl_msplit_count(bi_gemm_t h, int64_t M) {
  if (!h || M <= 0) return 0;
  int64_t s = h->num_sms / ((M + 63) / 64);
  s = std::max<int64_t>(1, std::min<int64_t>(s, h->kblocks));
  return int(s);
}

BI_CTL_API int bi_ctl_run_msplit(bi_gemm_t h, const void* x, int64_t M, const void* W,
                                 const bi_gemm_scales* scales, void* y, void* stream) {
  int rc = validate_run(h, x, M, W, scales, y);
  if (rc != BI_GEMM_OK || M == 0) return rc;
  std::lock_guard<std::mutex> lk(h->mu);
  return launch(h, x, M, W, scales, y, static_cast<cudaStream_t>(stream),
                bi_ctl_msplit_count(h, M), 0u);
}

// N2: M <= 16 goes to the CUDA-core kernel above; larger M to the product kernel.
BI_CTL_API int bi_ctl_run_smallm_fork(bi_gemm_t h, const void* x, int64_t M, const void* W,
                                      void* y, void* stream) {
  int rc = validate_run(h, x, M, W, nullptr, y);
  if (rc != BI_GEMM_OK || M == 0) return rc;
  if (h->dtype == BI_MXFP8E4M3_OUT_BF16) return BI_GEMM_ERR_UNSUPPORTED;
  if (M > 16) return bi_gemm_run(h, x, M, W, nullptr, y, stream);
  dim3 grid(unsigned((h->N + 127) / 128), unsigned(M));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->dtype == BI_BF16_OUT_F32)
    small_m_fma_kernel<true><<<grid, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                   static_cast<const __nv_bfloat16*>(W), y, int(M),
                                                   int(h->N), int(h->K));
  else
    small_m_fma_kernel<false><<<grid, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                                    static_cast<const __nv_bfloat16*>(W), y, int(M),
                                                    int(h->N), int(h->K));
  return cudaGetLastError() == cudaSuccess ? BI_GEMM_OK : BI_GEMM_ERR_CUDA;
}

// Failure injection: the producer withholds the first stage of each CTA's first tile, so the
// MMA issuer's bounded wait expires; the kernel must record BI_GEMM_ERR_TIMEOUT, drain, free
// its tensor memory and return, leaving the context usable.
BI_CTL_API int bi_ctl_run_stall(bi_gemm_t h, const void* x, int64_t M, const void* W,
                                const bi_gemm_scales* scales, void* y, void* stream) {
  int rc = validate_run(h, x, M, W, scales, y);
  if (rc != BI_GEMM_OK || M == 0) return rc;
  std::lock_guard<std::mutex> lk(h->mu);
  return launch(h, x, M, W, scales, y, static_cast<cudaStream_t>(stream), 0, 1u);
}

// Failure injection for the shared split-K merge: split 0 of every tile never counts its
// arrival, so the other split CTAs' bounded waits for it expire; the kernel must record
// BI_GEMM_ERR_TIMEOUT and return, and the next run must reset the arrival counters.
BI_CTL_API int bi_ctl_run_skip_arrival(bi_gemm_t h, const void* x, int64_t M, const void* W,
                                       const bi_gemm_scales* scales, void* y, void* stream) {
  int rc = validate_run(h, x, M, W, scales, y);
  if (rc != BI_GEMM_OK || M == 0) return rc;
  std::lock_guard<std::mutex> lk(h->mu);
  return launch(h, x, M, W, scales, y, static_cast<cudaStream_t>(stream), 0, 2u);
}

// Control N3 (RMSNorm): fp32 output (the values before the bf16 rounding, so that any change of
// reduction order shows) with the threads per row either fixed from d, the product's rule
// (mkeyed = 0), or chosen from the batch size as a library keyed on occupancy would: 1024 threads
// per row while M <= 16, 128 above (mkeyed = 1; a different butterfly and warp order).
BI_CTL_API int bi_ctl_rmsnorm_f32(const void* x, int64_t M, int64_t d, const void* g, float eps, void* y,
                                  int32_t mkeyed, void* stream) {
  if (M < 0 || !birms::valid_d(d) || !(eps >= 0.0f)) return BI_GEMM_ERR_INVALID_ARG;
  if (M == 0) return BI_GEMM_OK;
  if (!x || !g || !y) return BI_GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(y)) & 15u)
    return BI_GEMM_ERR_ALIGNMENT;
  const int nvec = int(d / birms::kVecElems);
  int threads = birms::threads_for(d);
  if (mkeyed) threads = std::max(threads, M <= 16 ? birms::kMaxThreads : birms::kMinThreads);
  if (nvec > threads * birms::kVecsPerThread) return BI_GEMM_ERR_UNSUPPORTED;
  birms::Params p;
  p.x = static_cast<const uint4*>(x);
  p.g = static_cast<const uint4*>(g);
  p.y = y;
  p.M = M;
  p.nvec = nvec;
  p.d = float(d);
  p.eps = eps;
  const unsigned grid = unsigned(std::min<int64_t>(M, 1024));
  birms::rmsnorm_kernel<true><<<grid, unsigned(threads), 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? BI_GEMM_OK : BI_GEMM_ERR_CUDA;
}

// This library's own copies of the attention entry points (the product's are hidden here).
BI_CTL_API int bi_ctl_attention_create(bi_attention_t* out, int64_t num_q_heads, int64_t num_kv_heads,
                                       int64_t head_dim, int64_t page_size, float scale, int64_t split_size) {
  return bi_attention_create(out, num_q_heads, num_kv_heads, head_dim, page_size, scale, split_size);
}

BI_CTL_API int bi_ctl_attention_run(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                                    const int32_t* q_pos, const void* k_cache, const void* v_cache,
                                    int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                                    int64_t max_pages, int64_t max_pos, void* o, void* stream) {
  return bi_attention_run(h, q, T, q_seq, q_pos, k_cache, v_cache, num_pages, page_table, num_seqs, max_pages,
                          max_pos, o, stream);
}

BI_CTL_API int bi_ctl_attention_get_device_error(bi_attention_t h, void* stream) {
  return bi_attention_get_device_error(h, stream);
}

BI_CTL_API int bi_ctl_attention_destroy(bi_attention_t h) { return bi_attention_destroy(h); }

BI_CTL_API int bi_ctl_attention_stall(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                                      const int32_t* q_pos, const void* k_cache, const void* v_cache,
                                      int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                                      int64_t max_pages, int64_t max_pos, void* o, uint64_t timeout_ns,
                                      void* stream) {
  if (!h) return BI_GEMM_ERR_INVALID_ARG;
  if (!h->tma || timeout_ns == 0) return BI_GEMM_ERR_UNSUPPORTED;
  return attention_run(h, q, T, q_seq, q_pos, k_cache, v_cache, num_pages, page_table, num_seqs, max_pages, max_pos, o,
                       stream, 0, timeout_ns, 1);
}

BI_CTL_API int bi_ctl_attention_run_kernel(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                                           const int32_t* q_pos, const void* k_cache, const void* v_cache,
                                           int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                                           int64_t max_pages, int64_t max_pos, void* o, int32_t kernel,
                                           void* stream) {
  if (!h || kernel < 1 || kernel > 2) return BI_GEMM_ERR_INVALID_ARG;
  if (kernel == 1 && !h->tma) return BI_GEMM_ERR_UNSUPPORTED;
  return attention_run(h, q, T, q_seq, q_pos, k_cache, v_cache, num_pages, page_table, num_seqs, max_pages, max_pos, o,
                       stream, -1, biattn::kTimeoutNs, kernel);
}
