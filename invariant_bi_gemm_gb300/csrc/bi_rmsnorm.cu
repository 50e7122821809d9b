// bi_rmsnorm.cu — batch-invariant RMSNorm for sm_103a.  Implements include/bi_rmsnorm.h.
//
// Definition ("Batch-invariant RMSNorm", nondeterminism article): per row,
// r = 1 / sqrt(sum_j x_j^2 / d + eps) and y_j = (x_j * r) * g_j, in fp32, rounded to bf16.
// Strategy (the article's data-parallel one): one thread block owns a row's whole reduction.
// The block size and each thread's share of the row are fixed from d alone, so the order of
// every floating-point operation on a row is the same for every M and whichever block runs it:
//   1. thread t sums x^2 over its vectors t, t + T, t + 2T, ... (T threads, 8 bf16 per 16-byte
//      vector), vectors in ascending order, elements in ascending column order, by fmaf;
//   2. the warp combines its 32 partials by an xor butterfly (offsets 16, 8, 4, 2, 1);
//   3. the T/32 warp partials are added in warp order, ((w0 + w1) + w2) + ...;
//   4. mean = sum / d (correctly rounded division), r = correctly rounded 1/sqrt(mean + eps);
//   5. y = bf16_rn((x * r) * g).
// The kernel is HBM-bound (each row read once, written once): 16-byte streaming loads,
// coalesced 16-byte stores and a programmatic dependent launch so that back-to-back kernels
// overlap their launch latency.  Two builds of the same arithmetic: a persistent grid of
// resident blocks striding over the rows, which loads a block's next row while it reduces the
// current one, and a build without that prefetch capped at half the registers, so that twice as
// many blocks fit on an SM; when the rows outnumber the first build's resident blocks but not the
// second's, the second runs and every row has a block of its own.  Which build runs depends on
// M; no operation on a row does.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/bi_rmsnorm.h"

#ifndef BI_GEMM_API
#define BI_GEMM_API extern "C" __attribute__((visibility("default")))
#endif

namespace birms {

constexpr int kVecElems = 8;        // bf16 per 16-byte vector
constexpr int kVecsPerThread = 4;   // vectors per thread at most
constexpr int kMinThreads = 128;
constexpr int kMaxThreads = 1024;
constexpr int64_t kMaxD = int64_t(kMaxThreads) * kVecsPerThread * kVecElems;   // 32768

struct Params {
  const uint4* x;
  const uint4* g;
  void* y;
  int64_t M;
  int32_t nvec;      // 16-byte vectors per row (d / 8)
  float d;           // row length as fp32 (exact: d <= 32768)
  float eps;
};

// 16-byte load that does not allocate in L1 (each x byte is read once).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float sum_squares(float s, uint32_t w) {
  const float a = bf16_lo(w), b = bf16_hi(w);
  s = __fmaf_rn(a, a, s);
  return __fmaf_rn(b, b, s);
}

__device__ __forceinline__ float scaled(float x, float g, float r) { return __fmul_rn(__fmul_rn(x, r), g); }

__device__ __forceinline__ uint32_t scale_pair(uint32_t xw, uint32_t gw, float r) {
  return pack_bf16x2(scaled(bf16_lo(xw), bf16_lo(gw), r), scaled(bf16_hi(xw), bf16_hi(gw), r));
}

// kOutF32 (test builds only): store the fp32 values before the bf16 rounding.  kPrefetch: the
// persistent build (a block's next row is loaded while the current one is reduced).
template <bool kOutF32, bool kPrefetch = true>
__global__ void __launch_bounds__(kMaxThreads, kPrefetch ? 1 : 2) rmsnorm_kernel(const Params p) {
  __shared__ float partial[2][kMaxThreads / 32];
  const int T = int(blockDim.x);
  const int t = int(threadIdx.x);
  const int lane = t & 31, warp = t >> 5, nwarps = T >> 5;

  uint4 cur[kVecsPerThread], nxt[kPrefetch ? kVecsPerThread : 1];
  auto load_row = [&](int64_t row, uint4 (&dst)[kVecsPerThread]) {
    const uint4* src = p.x + row * p.nvec;
#pragma unroll
    for (int j = 0; j < kVecsPerThread; ++j) {
      const int v = j * T + t;
      if (v < p.nvec) dst[j] = ld_stream(src + v);
    }
  };

  // Programmatic dependent launch: this block may start while the previous kernel in the stream
  // finishes; it waits for that kernel (and its memory) before the first global access, and lets
  // the next kernel start its own launch as soon as every block of this one is running.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  int64_t row = blockIdx.x;
  if (row < p.M) load_row(row, cur);
  int buf = 0;
  for (; row < p.M; row += gridDim.x) {
    const int64_t next = row + gridDim.x;
    if constexpr (kPrefetch) {
      if (next < p.M) load_row(next, nxt);   // in flight while this row is reduced
    }

    // 1. this thread's squares, vectors and elements in ascending order
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kVecsPerThread; ++j) {
      if (j * T + t < p.nvec) {
        s = sum_squares(s, cur[j].x);
        s = sum_squares(s, cur[j].y);
        s = sum_squares(s, cur[j].z);
        s = sum_squares(s, cur[j].w);
      }
    }
    // 2. fixed butterfly within the warp (every lane ends with the same value)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xFFFFFFFFu, s, o));
    // 3. warp partials in warp order (double-buffered: one barrier per row suffices)
    if (lane == 0) partial[buf][warp] = s;
    __syncthreads();
    float total = partial[buf][0];
    for (int w = 1; w < nwarps; ++w) total = __fadd_rn(total, partial[buf][w]);
    // 4. mean and reciprocal square root, both correctly rounded
    const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(total, p.d), p.eps));
    // 5. scale, weight, round, store
#pragma unroll
    for (int j = 0; j < kVecsPerThread; ++j) {
      const int v = j * T + t;
      if (v < p.nvec) {
        const uint4 gv = __ldg(p.g + v);
        if constexpr (kOutF32) {
          float4* dst = static_cast<float4*>(p.y) + (row * p.nvec + v) * 2;
          dst[0] = make_float4(scaled(bf16_lo(cur[j].x), bf16_lo(gv.x), r), scaled(bf16_hi(cur[j].x), bf16_hi(gv.x), r),
                               scaled(bf16_lo(cur[j].y), bf16_lo(gv.y), r), scaled(bf16_hi(cur[j].y), bf16_hi(gv.y), r));
          dst[1] = make_float4(scaled(bf16_lo(cur[j].z), bf16_lo(gv.z), r), scaled(bf16_hi(cur[j].z), bf16_hi(gv.z), r),
                               scaled(bf16_lo(cur[j].w), bf16_lo(gv.w), r), scaled(bf16_hi(cur[j].w), bf16_hi(gv.w), r));
        } else {
          uint4 o;
          o.x = scale_pair(cur[j].x, gv.x, r);
          o.y = scale_pair(cur[j].y, gv.y, r);
          o.z = scale_pair(cur[j].z, gv.z, r);
          o.w = scale_pair(cur[j].w, gv.w, r);
          static_cast<uint4*>(p.y)[row * p.nvec + v] = o;
        }
      }
    }
    if constexpr (kPrefetch) {
#pragma unroll
      for (int j = 0; j < kVecsPerThread; ++j) cur[j] = nxt[j];
    } else if (next < p.M) {
      load_row(next, cur);
    }
    buf ^= 1;
  }
}

// Threads per row: enough that each owns at most kVecsPerThread vectors, a multiple of 32,
// at least kMinThreads.  A function of d only.
inline int threads_for(int64_t d) {
  const int nvec = int(d / kVecElems);
  int threads = (nvec + kVecsPerThread - 1) / kVecsPerThread;
  threads = (threads + 31) / 32 * 32;
  return std::min(kMaxThreads, std::max(kMinThreads, threads));
}

inline bool valid_d(int64_t d) { return d >= kVecElems && d <= kMaxD && d % kVecElems == 0; }

}  // namespace birms

struct bi_rmsnorm {
  int64_t d = 0;
  float eps = 0.0f;
  int device = 0;
  int threads = 0;
  int vecs_per_thread = 0;
  int max_ctas = 0;          // resident blocks of the persistent build
  int max_ctas_single = 0;   // resident blocks of the one-row-per-block build
  int num_sms = 0;
};

BI_GEMM_API int bi_rmsnorm_create(bi_rmsnorm_t* out, int64_t d, float eps) {
  if (!out) return BI_GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!std::isfinite(eps) || eps < 0.0f) return BI_GEMM_ERR_INVALID_ARG;
  if (!birms::valid_d(d)) return BI_GEMM_ERR_UNSUPPORTED;
  const int nvec = int(d / birms::kVecElems);
  const int threads = birms::threads_for(d);

  int dev = 0, major = 0, minor = 0, sms = 0, per_sm = 0, per_sm_single = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return BI_GEMM_ERR_UNSUPPORTED;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, birms::rmsnorm_kernel<false, true>, threads, 0) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_single, birms::rmsnorm_kernel<false, false>, threads,
                                                    0) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  bi_rmsnorm* h = new (std::nothrow) bi_rmsnorm();
  if (!h) return BI_GEMM_ERR_OOM;
  h->d = d;
  h->eps = eps;
  h->device = dev;
  h->threads = threads;
  h->vecs_per_thread = (nvec + threads - 1) / threads;
  h->num_sms = sms;
  h->max_ctas = std::max(1, per_sm) * sms;
  h->max_ctas_single = std::max(1, per_sm_single) * sms;
  *out = h;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_rmsnorm_run(bi_rmsnorm_t h, const void* x, int64_t M, const void* g, void* y,
                               void* stream) {
  if (!h || M < 0) return BI_GEMM_ERR_INVALID_ARG;
  if (M == 0) return BI_GEMM_OK;
  if (!x || !g || !y) return BI_GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(y)) & 15u)
    return BI_GEMM_ERR_ALIGNMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (dev != h->device) return BI_GEMM_ERR_INVALID_ARG;
  birms::Params p;
  p.x = static_cast<const uint4*>(x);
  p.g = static_cast<const uint4*>(g);
  p.y = y;
  p.M = M;
  p.nvec = int32_t(h->d / birms::kVecElems);
  p.d = float(h->d);
  p.eps = h->eps;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  // Rows that outnumber the persistent build's resident blocks but not the single-row build's:
  // every row its own block (the persistent build would give some blocks two rows in turn).
  // Fewer rows run the persistent build, one row per block too, without its register cap.
  const bool single = M > h->max_ctas && M <= h->max_ctas_single;
  cfg.gridDim = dim3(unsigned(single ? M : std::min<int64_t>(M, h->max_ctas)));
  cfg.blockDim = dim3(unsigned(h->threads));
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, single ? birms::rmsnorm_kernel<false, false> : birms::rmsnorm_kernel<false, true>,
                         p) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_rmsnorm_get_config(bi_rmsnorm_t h, bi_rmsnorm_config* c) {
  if (!h || !c) return BI_GEMM_ERR_INVALID_ARG;
  c->d = int32_t(h->d);
  c->threads = h->threads;
  c->vectors_per_thread = h->vecs_per_thread;
  c->max_ctas = h->max_ctas;
  c->num_sms = h->num_sms;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_rmsnorm_destroy(bi_rmsnorm_t h) {
  delete h;
  return BI_GEMM_OK;
}
