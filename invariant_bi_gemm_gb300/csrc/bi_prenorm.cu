// bi_prenorm.cu — batch-invariant pre-norm projection of the hyper-connection (mHC) block,
// sm_103a.  Implements include/bi_prenorm.h.
//
// y[i, :] = (x[i, :] . W) / sqrt(sum_k x[i, k]^2 / K + eps), the pre-norm GEMM with its fused
// RMSNorm of "[BI][DSv4] Make mHC tilelang ops batch invariant", with the K split fixed per
// handle (chunks of `chunk` elements) instead of derived from the token count.
//   one block per (chunk, 16-row tile): the chunk of x (16 rows) and of W staged with
//     cp.async (rows padded so that ldmatrix reads are free of bank conflicts); warp w computes
//     columns 8w..8w+7 of the tile's projection with mma.sync m16n8k16 (bf16, fp32 accumulate,
//     k ascending); every row's sum of squares as eight runs of chunk/8 elements (fma, ascending),
//     combined by a fixed xor butterfly; both written per chunk;
//   a merge kernel (one block per row, launched as a programmatic dependent so that its launch
//     overlaps the chunk kernel): per output, the chunks' projections and sums of squares added
//     in ascending chunk order, r = 1/sqrt(ss / K + eps) correctly rounded, y = projection * r.
// Nothing in the arithmetic of row i reads another row or M.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/bi_prenorm.h"
#include "ptx.cuh"

#ifndef BI_GEMM_API
#define BI_GEMM_API extern "C" __attribute__((visibility("default")))
#endif

namespace biprn {

namespace ptx = bigemm::ptx;

constexpr int kThreads = 128;      // four warps: one per 8-column n tile of the projection
constexpr int kRows = 16;          // rows of x per block (the MMA's M)
constexpr int kDefaultChunk = 512;
constexpr int kMergeThreads = 256;

struct Params {
  const uint16_t* x;   // [M, K]
  const uint16_t* w;   // [K, N]
  float* y;            // [M, N]
  float* part;         // [S, M, N] per-chunk projections
  float* ssp;          // [S, M] per-chunk sums of squares
  int64_t M;
  int32_t K, N, chunk, S;
  float eps;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d += a * b: a 16 x 16 (row-major, bf16), b 16 x 8 (column-major, bf16), d 16 x 8 fp32.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Staged strides (bytes): rows shift by an odd number of 16-byte bank groups.
__host__ __device__ inline int x_stride(int chunk) { return chunk * 2 + 16; }
__host__ __device__ inline int w_stride(int N) { return (N * 2 / 16) % 2 == 0 ? N * 2 + 16 : N * 2; }
inline size_t smem_bytes(int chunk, int N) { return size_t(kRows) * x_stride(chunk) + size_t(chunk) * w_stride(N); }

__global__ void __launch_bounds__(kThreads) chunk_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int XS = x_stride(p.chunk), WS = w_stride(p.N);
  uint8_t* xs = smem;
  uint8_t* ws = smem + kRows * XS;
  const uint32_t xs_a = ptx::smem_u32(xs), ws_a = ptx::smem_u32(ws);
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int s = int(blockIdx.x);
  const int64_t row0 = int64_t(blockIdx.y) * kRows;
  const int32_t k0 = s * p.chunk;
  // launched as a programmatic dependent: x may be the previous kernel's output and the
  // workspace its input, so nothing global is touched before that kernel has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // stage the chunk: x rows (zeros past M or K) and W rows (zeros past K), 16-byte pieces
  const int xc = p.chunk / 8;   // pieces per x row
  for (int i = tid; i < kRows * xc; i += kThreads) {
    const int r = i / xc, c = i - r * xc;
    const int32_t k = k0 + c * 8;
    const bool ok = row0 + r < p.M && k < p.K;
    ptx::cp_async_16(xs_a + r * XS + c * 16, ok ? static_cast<const void*>(p.x + (row0 + r) * p.K + k) : p.x,
                     ok ? 16u : 0u);
  }
  const int wc = p.N / 8;       // pieces per W row
  for (int i = tid; i < p.chunk * wc; i += kThreads) {
    const int r = i / wc, c = i - r * wc;
    const bool ok = k0 + r < p.K;
    ptx::cp_async_16(ws_a + r * WS + c * 16, ok ? static_cast<const void*>(p.w + int64_t(k0 + r) * p.N + c * 8) : p.w,
                     ok ? 16u : 0u);
  }
  ptx::cp_async_commit();
  ptx::cp_async_wait<0>();
  __syncthreads();

  // projection: this warp's n tile, all k steps of the chunk in ascending order
  if (warp < p.N / 8) {
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int m = lane >> 3, r8 = lane & 7;
    for (int ks = 0; ks < p.chunk / 16; ks += 2) {
      uint32_t a0[4], a1[4], b[4];
      // A: rows (m & 1) * 8 + r8, k = 16 ks + (m >> 1) * 8 (and the next k step)
      ldsm_x4(xs_a + ((m & 1) * 8 + r8) * XS + (16 * ks + (m >> 1) * 8) * 2, a0);
      ldsm_x4(xs_a + ((m & 1) * 8 + r8) * XS + (16 * (ks + 1) + (m >> 1) * 8) * 2, a1);
      // B: k rows 16 ks + 8 m + r8 (four 8-row blocks: two k steps), columns 8 warp .. + 7
      ldsm_x4_trans(ws_a + (16 * ks + 8 * m + r8) * WS + warp * 16, b);
      mma16816(d, a0, b[0], b[1]);
      mma16816(d, a1, b[2], b[3]);
    }
    const int g = lane >> 2, t = lane & 3, col = warp * 8 + 2 * t;
    if (row0 + g < p.M)
      *reinterpret_cast<float2*>(p.part + (int64_t(s) * p.M + row0 + g) * p.N + col) = make_float2(d[0], d[1]);
    if (row0 + g + 8 < p.M)
      *reinterpret_cast<float2*>(p.part + (int64_t(s) * p.M + row0 + g + 8) * p.N + col) = make_float2(d[2], d[3]);
  }

  // sums of squares: thread (row tid / 8, run tid % 8) over chunk / 8 elements, then a fixed
  // butterfly over the eight runs (every lane of the eight ends with the same value)
  {
    const int r = tid >> 3, e = tid & 7, len = p.chunk / 8;
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs + r * XS + e * len * 2);
    float ss = 0.0f;
    for (int i = 0; i < len / 2; ++i) {
      const uint32_t v = xr[i];
      ss = __fmaf_rn(bf16_lo(v), bf16_lo(v), ss);
      ss = __fmaf_rn(bf16_hi(v), bf16_hi(v), ss);
    }
    ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, 4));
    ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, 2));
    ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, 1));
    if (e == 0 && row0 + r < p.M) p.ssp[int64_t(s) * p.M + row0 + r] = ss;
  }

  // the merge kernel (launched as a programmatic dependent) may start its launch now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Merge, one block per row: the chunks' projections and sums of squares in ascending chunk
// order.  Thread (c, e) of a batch loads group e (four outputs) of chunk s0 + c into shared
// memory, so a batch is one round of independent loads; threads e < N / 4 then add them in order.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const Params p) {
  __shared__ float4 buf[kMergeThreads];
  __shared__ float sbuf[kMergeThreads];
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the chunk kernel's results are complete
  const int tid = int(threadIdx.x);
  const int64_t row = blockIdx.x;
  const int nq = p.N / 4;
  const int per = kMergeThreads / nq;           // chunks per batch
  const int c = tid / nq, e = tid - c * nq;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float ss = 0.0f;
  for (int s0 = 0; s0 < p.S; s0 += per) {
    const int nb = min(per, p.S - s0);
    if (c < nb) {
      buf[tid] = reinterpret_cast<const float4*>(p.part + (int64_t(s0 + c) * p.M + row) * p.N)[e];
      if (e == 0) sbuf[c] = p.ssp[int64_t(s0 + c) * p.M + row];
    }
    __syncthreads();
    if (tid < nq) {
      for (int j = 0; j < nb; ++j) {
        const float4 v = buf[j * nq + tid];
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
        ss = __fadd_rn(ss, sbuf[j]);
      }
    }
    __syncthreads();
  }
  if (tid < nq) {
    const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, float(p.K)), p.eps));
    float* yr = p.y + row * p.N + 4 * tid;
    yr[0] = __fmul_rn(acc.x, rr);
    yr[1] = __fmul_rn(acc.y, rr);
    yr[2] = __fmul_rn(acc.z, rr);
    yr[3] = __fmul_rn(acc.w, rr);
  }
}

}  // namespace biprn

struct bi_prenorm {
  int K = 0, N = 0, chunk = 0, S = 0;
  float eps = 0.0f;
  int device = 0;
  size_t smem = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

BI_GEMM_API int bi_prenorm_create(bi_prenorm_t* out, int64_t K, int64_t N, float eps, int64_t chunk) {
  if (!out) return BI_GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!std::isfinite(eps) || eps < 0.0f || chunk < 0) return BI_GEMM_ERR_INVALID_ARG;
  const int64_t ch = chunk ? chunk : biprn::kDefaultChunk;
  if (K < 8 || K % 8 != 0 || K >= (int64_t(1) << 24) || N < 8 || N > 32 || N % 8 != 0 || ch % 64 != 0 ||
      ch > 1024)
    return BI_GEMM_ERR_UNSUPPORTED;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return BI_GEMM_ERR_UNSUPPORTED;
  const size_t smem = biprn::smem_bytes(int(ch), int(N));
  // the attribute is per kernel and shared by all handles: set the largest any handle can need
  if (cudaFuncSetAttribute(biprn::chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(biprn::smem_bytes(1024, 32))) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  bi_prenorm* h = new (std::nothrow) bi_prenorm();
  if (!h) return BI_GEMM_ERR_OOM;
  h->K = int(K);
  h->N = int(N);
  h->chunk = int(ch);
  h->S = int((K + ch - 1) / ch);
  h->eps = eps;
  h->device = dev;
  h->smem = smem;
  *out = h;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_prenorm_run(bi_prenorm_t h, const void* x, int64_t M, const void* W, float* y, void* stream) {
  if (!h || M < 0) return BI_GEMM_ERR_INVALID_ARG;
  if (M == 0) return BI_GEMM_OK;
  if (!x || !W || !y) return BI_GEMM_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W)) & 15u) || (reinterpret_cast<uintptr_t>(y) & 7u))
    return BI_GEMM_ERR_ALIGNMENT;
  if ((M + biprn::kRows - 1) / biprn::kRows > 65535 || M >= (int64_t(1) << 31) || M * h->N >= (int64_t(1) << 31))
    return BI_GEMM_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (dev != h->device) return BI_GEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t part = (size_t(h->S) * M * h->N * sizeof(float) + 255) & ~size_t(255);
  const size_t need = part + size_t(h->S) * M * sizeof(float);
  if (need > h->ws_bytes) {
    if (h->ws) cudaFreeAsync(h->ws, st);
    h->ws = nullptr;
    h->ws_bytes = 0;
    void* p = nullptr;
    if (cudaMallocAsync(&p, need, st) != cudaSuccess) {
      cudaGetLastError();
      return BI_GEMM_ERR_OOM;
    }
    h->ws = p;
    h->ws_bytes = need;
  }
  biprn::Params p;
  std::memset(&p, 0, sizeof(p));
  p.x = static_cast<const uint16_t*>(x);
  p.w = static_cast<const uint16_t*>(W);
  p.y = y;
  p.part = static_cast<float*>(h->ws);
  p.ssp = reinterpret_cast<float*>(static_cast<uint8_t*>(h->ws) + part);
  p.M = M;
  p.K = h->K;
  p.N = h->N;
  p.chunk = h->chunk;
  p.S = h->S;
  p.eps = h->eps;
  // Both kernels are programmatic dependents of the kernel before them: each launches while
  // that kernel finishes and waits for it (griddepcontrol.wait) before touching global memory.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cc;
  std::memset(&cc, 0, sizeof(cc));
  cc.gridDim = dim3(unsigned(h->S), unsigned((M + biprn::kRows - 1) / biprn::kRows));
  cc.blockDim = dim3(biprn::kThreads);
  cc.dynamicSmemBytes = h->smem;
  cc.stream = st;
  cc.attrs = attr;
  cc.numAttrs = 1;
  if (cudaLaunchKernelEx(&cc, biprn::chunk_kernel, p) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(unsigned(M));
  cfg.blockDim = dim3(biprn::kMergeThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, biprn::merge_kernel, p) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return BI_GEMM_ERR_CUDA;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_prenorm_get_config(bi_prenorm_t h, bi_prenorm_config* c) {
  if (!h || !c) return BI_GEMM_ERR_INVALID_ARG;
  c->K = h->K;
  c->N = h->N;
  c->chunk = h->chunk;
  c->splits = h->S;
  c->tile_rows = biprn::kRows;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_prenorm_destroy(bi_prenorm_t h) {
  if (!h) return BI_GEMM_OK;
  if (h->ws) cudaFree(h->ws);
  delete h;
  return BI_GEMM_OK;
}
