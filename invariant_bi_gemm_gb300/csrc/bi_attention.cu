// bi_attention.cu — batch-invariant decode attention over a paged KV cache, sm_103a.
// Implements include/bi_attention.h.
//
// "Batch-invariant attention" (nondeterminism article): split the keys of a query at a fixed
// split SIZE, reduce each split in one fixed order, merge the splits in a fixed order.  The
// work unit is (query token t, KV head kh, split s); one block of 128 threads runs a unit:
//   1. the G query heads of kh are widened to fp32 in shared memory;
//   2. the split's keys, then its values, stream through a 3-deep ring of 128-position stages
//      (cp.async, 16-byte chunks, row-XOR swizzle so that both passes read without bank
//      conflicts); rows past p, or of an invalid page, are zero-filled and masked;
//   3. pass 1: thread r owns position r of a key stage and computes its G scores as fp32 dot
//      products in ascending dimension (fmaf), times scale * log2(e);
//   4. per head, the split's maximum m (exact, order-free) and weights w_j = exp2(s_j - m);
//   5. pass 2: each thread owns G*D/128 consecutive outputs of one head and accumulates
//      acc += w_j v_j and l += w_j over the split's positions in ascending order;
//   6. a single-split token writes bf16(acc / l); otherwise the unit stores (m, l, acc) and the
//      last of the token's split blocks to arrive (an integer counter) merges all splits in
//      ascending s: M = max m_s, L = sum l_s 2^(m_s - M), A = sum acc_s 2^(m_s - M), o = A / L.
//      A single split merged this way gives the same bits as the direct path (2^0 = 1).
// A plan kernel first turns q_pos into per-token unit offsets (a prefix sum) and the token of
// every unit, and zeroes the counters.  The attention kernel is persistent: a block fetches its
// next unit's coordinates, page indices and query while it works on the current one and issues
// the next unit's first stages into the ring during the current unit's last ones, so that the
// key/value stream does not drain between units.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/bi_attention.h"
#include "ptx.cuh"

#ifndef BI_GEMM_API
#define BI_GEMM_API extern "C" __attribute__((visibility("default")))
#endif

namespace biattn {

namespace ptx = bigemm::ptx;

constexpr int kThreads = 128;        // threads per block = positions per stage
constexpr int kStages = 3;           // staging ring depth
constexpr int kDefaultSplit = 256;
constexpr uint32_t kErrInput = 1u;   // bad q_seq / q_pos / page-table extent
constexpr uint32_t kErrPage = 2u;    // page index outside [0, num_pages)
constexpr uint32_t kErrBound = 4u;   // q_pos above the host's max_pos

struct Params {
  const uint16_t* q;
  const int32_t* q_seq;
  const int32_t* q_pos;
  const uint16_t* kc;
  const uint16_t* vc;
  const int32_t* table;
  uint16_t* o;
  int32_t* cum;      // [T + 1] first unit of each token
  int32_t* umap;     // [units] the token of each unit
  uint32_t* cnt;     // [T * Hkv] merge counters
  float* part;       // [T * Hkv * max_splits, G, D] partial weighted sums
  float* ml;         // [T * Hkv * max_splits, G, 2] (maximum, sum of weights)
  uint32_t* status;
  int64_t T, num_pages, B, max_pages;
  int32_t Hq, Hkv, page_size, split, max_splits;
  int32_t pages_per_split;   // most pages one split can touch
  float c;           // scale * log2(e)
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f_bf16(float f) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.0f), "f"(f));
  return uint16_t(r & 0xFFFFu);
}

// Number of splits of a token at position p.
__device__ __forceinline__ int32_t splits_of(int32_t p, int32_t split) { return p / split + 1; }

// Unit offsets: cum[t] = Hkv * (splits of the tokens before t) and the token of every unit; a
// token with an input the kernel cannot serve gets no units (and sets the status word).  Also
// zeroes the merge counters.
__global__ void __launch_bounds__(1024) plan_kernel(const Params p) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < p.T; base += 1024) {
    const int64_t t = base + tid;
    int32_t n = 0;
    if (t < p.T) {
      const int32_t b = p.q_seq[t], pos = p.q_pos[t];
      if (b < 0 || b >= p.B || pos < 0 || int64_t(pos / p.page_size) >= p.max_pages) {
        atomicOr(p.status, kErrInput);
      } else if (splits_of(pos, p.split) > p.max_splits) {
        atomicOr(p.status, kErrBound);
      } else {
        n = splits_of(pos, p.split) * p.Hkv;
      }
      for (int kh = 0; kh < p.Hkv; ++kh) p.cnt[t * p.Hkv + kh] = 0u;
    }
    int32_t x = n;   // inclusive scan within the warp, then over the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int32_t w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int32_t incl = carry + x + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (t < p.T) {
      p.cum[t] = incl - n;
      for (int32_t i = incl - n; i < incl; ++i) p.umap[i] = int32_t(t);
    }
    __syncthreads();
    if (tid == 1023) carry = incl;
    __syncthreads();
  }
  if (tid == 0) p.cum[p.T] = carry;
}

template <int D, int G>
struct Cfg {
  static constexpr int CHUNKS = D / 8;                 // 16-byte chunks per row
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int STAGE_BYTES = kThreads * ROW_BYTES;
  static constexpr int OPT = (G * D) / kThreads >= 1 ? (G * D) / kThreads : 1;   // outputs per thread
  static constexpr int OUT_THREADS = G * D / OPT;
  static_assert(OPT == 1 || OPT == 2 || OPT == 4 || OPT == 8, "outputs per thread");
  static_assert(OUT_THREADS <= kThreads, "output threads");
  static size_t smem_bytes(int split, int pages_per_split) {
    return size_t(kStages) * STAGE_BYTES + sizeof(float) * (size_t(G) * D + size_t(G) * split + G * 4) +
           sizeof(int32_t) * 2 * size_t(pages_per_split);
  }
};

// Load OPT consecutive bf16 (at dimension d, a multiple of OPT) of a staged row as fp32.
template <int OPT>
__device__ __forceinline__ void load_piece(const uint8_t* p, float (&v)[OPT]) {
  if constexpr (OPT == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  } else if constexpr (OPT == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  } else if constexpr (OPT == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    v[0] = bf16_lo(w); v[1] = bf16_hi(w);
  } else {
    v[0] = bf16_f(*reinterpret_cast<const uint16_t*>(p));
  }
}

// One unit's coordinates, read from the plan.
struct Unit {
  int64_t t, b;
  int32_t kh, s, pos, nsplit, j0, valid, nsub, page0, npages;
};

__device__ __forceinline__ Unit unit_of(const Params& p, int64_t u) {
  Unit w;
  w.t = p.umap[u];
  const int32_t r = int32_t(u - p.cum[w.t]);
  w.s = r / p.Hkv;
  w.kh = r - w.s * p.Hkv;
  w.b = p.q_seq[w.t];
  w.pos = p.q_pos[w.t];
  w.nsplit = splits_of(w.pos, p.split);
  w.j0 = w.s * p.split;
  w.valid = min(p.split, w.pos + 1 - w.j0);                  // keys in this split (>= 1)
  w.nsub = (w.valid + kThreads - 1) / kThreads;
  w.page0 = w.j0 / p.page_size;
  w.npages = (w.j0 + w.valid - 1) / p.page_size - w.page0 + 1;
  return w;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) attn_kernel(const Params p) {
  using C = Cfg<D, G>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* qs = reinterpret_cast<float*>(smem + kStages * C::STAGE_BYTES);   // [G][D]
  float* sc = qs + G * D;                                                   // [G][split]
  float* red = sc + G * p.split;                                            // [G][4]
  int32_t* pages = reinterpret_cast<int32_t*>(red + G * 4);                 // [2][max_pages_per_split]
  __shared__ uint32_t s_last;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int og = (tid * C::OPT) / D, od = (tid * C::OPT) % D;   // pass-2 outputs: head, first dim
  const bool has_out = tid < C::OUT_THREADS;
  constexpr int QPT = G * D / kThreads >= 1 ? G * D / kThreads : 1;   // query elements per thread

  const int32_t total = p.cum[p.T];
  int64_t u = blockIdx.x;
  if (u >= total) return;

  // A unit's page indices go to its half of `pages`; its query heads, widened, to qs.
  auto fill_pages = [&](const Unit& w, int half) {
    for (int i = tid; i < w.npages; i += kThreads)
      pages[half * p.pages_per_split + i] = p.table[w.b * p.max_pages + w.page0 + i];
  };
  auto load_q = [&](const Unit& w, uint16_t (&qr)[QPT]) {
#pragma unroll
    for (int e = 0; e < QPT; ++e) {
      const int i = tid * QPT + e;
      qr[e] = i < G * D ? p.q[(w.t * p.Hq + int64_t(w.kh) * G) * D + i] : uint16_t(0);
    }
  };
  auto store_q = [&](const uint16_t (&qr)[QPT]) {
#pragma unroll
    for (int e = 0; e < QPT; ++e) {
      const int i = tid * QPT + e;
      if (i < G * D) qs[i] = bf16_f(qr[e]);
    }
  };

  bool bad_page = false;
  // Load number i of unit w (key stages, then value stages) into ring slot `slot`.
  auto issue = [&](const Unit& w, int half, int i, int slot) {
    const bool isv = i >= w.nsub;
    const int sub = isv ? i - w.nsub : i;
    const uint16_t* base = isv ? p.vc : p.kc;
    const uint32_t dst0 = ptx::smem_u32(ring + slot * C::STAGE_BYTES);
    const int32_t* pg = pages + half * p.pages_per_split;
#pragma unroll 4
    for (int it = 0; it < C::CHUNKS; ++it) {
      const int lin = it * kThreads + tid;
      const int row = lin / C::CHUNKS, c = lin % C::CHUNKS;
      const uint32_t dst = dst0 + row * C::ROW_BYTES + ((c ^ (row & (C::CHUNKS - 1))) << 4);
      const void* src = base;
      uint32_t bytes = 0;
      if (sub * kThreads + row < w.valid) {
        const int32_t j = w.j0 + sub * kThreads + row;
        const int64_t page = pg[j / p.page_size - w.page0];
        if (page >= 0 && page < p.num_pages) {
          src = base + ((page * p.page_size + j % p.page_size) * p.Hkv + w.kh) * D + c * 8;
          bytes = 16;
        } else {
          bad_page = true;
        }
      }
      ptx::cp_async_16(dst, src, bytes);   // bytes == 0: zero-fill, nothing read
    }
  };

  Unit cur = unit_of(p, u);
  int half = 0;
  {
    uint16_t qr[QPT];
    load_q(cur, qr);
    fill_pages(cur, half);
    store_q(qr);
  }
  __syncthreads();
  uint32_t seq = 0;   // sequence number of the next load to issue (its ring slot is seq % kStages)
  uint32_t cons = 0;  // sequence number of the next load to consume
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < 2 * cur.nsub) issue(cur, half, i, int(seq % kStages));
    ++seq;
    ptx::cp_async_commit();
  }

  while (true) {
    // the next unit of this block: its coordinates, pages and query are fetched now, so that
    // its first stages can be issued while this unit finishes
    const int64_t un = u + gridDim.x;
    const bool has_next = un < total;
    Unit nxt;
    uint16_t qn[QPT];
    if (has_next) {
      nxt = unit_of(p, un);
      fill_pages(nxt, half ^ 1);
      load_q(nxt, qn);
    }
    __syncthreads();   // the next unit's pages are visible to every issuing thread

    const int nload = 2 * cur.nsub;
    float acc[C::OPT];
#pragma unroll
    for (int e = 0; e < C::OPT; ++e) acc[e] = 0.0f;
    float l = 0.0f;
    for (int i = 0; i < nload; ++i) {
      const int ahead = i + kStages - 1;   // the load issued now: this unit's, or the next's
      if (ahead < nload) issue(cur, half, ahead, int(seq % kStages));
      else if (has_next && ahead - nload < 2 * nxt.nsub) issue(nxt, half ^ 1, ahead - nload, int(seq % kStages));
      ++seq;
      ptx::cp_async_commit();
      ptx::cp_async_wait<kStages - 1>();
      __syncthreads();
      const uint8_t* buf = ring + (cons % kStages) * C::STAGE_BYTES;
      ++cons;
      if (i < cur.nsub) {
        // pass 1: the scores of position jl for the G heads
        const int row = tid, jl = i * kThreads + row;
        if (jl < cur.valid) {
          float dot[G];
#pragma unroll
          for (int g = 0; g < G; ++g) dot[g] = 0.0f;
#pragma unroll 4
          for (int c = 0; c < C::CHUNKS; ++c) {
            float kf[8];
            load_piece<8>(buf + row * C::ROW_BYTES + ((c ^ (row & (C::CHUNKS - 1))) << 4), kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float4 q0 = *reinterpret_cast<const float4*>(qs + g * D + c * 8);
              const float4 q1 = *reinterpret_cast<const float4*>(qs + g * D + c * 8 + 4);
              dot[g] = __fmaf_rn(q0.x, kf[0], dot[g]);
              dot[g] = __fmaf_rn(q0.y, kf[1], dot[g]);
              dot[g] = __fmaf_rn(q0.z, kf[2], dot[g]);
              dot[g] = __fmaf_rn(q0.w, kf[3], dot[g]);
              dot[g] = __fmaf_rn(q1.x, kf[4], dot[g]);
              dot[g] = __fmaf_rn(q1.y, kf[5], dot[g]);
              dot[g] = __fmaf_rn(q1.z, kf[6], dot[g]);
              dot[g] = __fmaf_rn(q1.w, kf[7], dot[g]);
            }
          }
#pragma unroll
          for (int g = 0; g < G; ++g) sc[g * p.split + jl] = __fmul_rn(dot[g], p.c);
        }
        if (i == cur.nsub - 1) {
          // the split's maximum per head, then the weights in place
          __syncthreads();
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float m = -INFINITY;
            for (int jj = tid; jj < cur.valid; jj += kThreads) m = fmaxf(m, sc[g * p.split + jj]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if (lane == 0) red[g * 4 + warp] = m;
          }
          __syncthreads();
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float m = fmaxf(fmaxf(red[g * 4 + 0], red[g * 4 + 1]), fmaxf(red[g * 4 + 2], red[g * 4 + 3]));
            for (int jj = tid; jj < cur.valid; jj += kThreads)
              sc[g * p.split + jj] = exp2f(__fsub_rn(sc[g * p.split + jj], m));
          }
        }
      } else if (has_out) {
        // pass 2: weighted sum of the value rows of this stage, ascending position
        const int sub = i - cur.nsub;
        const int rows = min(kThreads, cur.valid - sub * kThreads);
        const float* w = sc + og * p.split + sub * kThreads;
        const int chunk = od / 8, within = (od % 8) * 2;
#pragma unroll 4
        for (int row = 0; row < rows; ++row) {
          float v[C::OPT];
          load_piece<C::OPT>(buf + row * C::ROW_BYTES + ((chunk ^ (row & (C::CHUNKS - 1))) << 4) + within, v);
          const float wj = w[row];
#pragma unroll
          for (int e = 0; e < C::OPT; ++e) acc[e] = __fmaf_rn(wj, v[e], acc[e]);
          l = __fadd_rn(l, wj);
        }
      }
      __syncthreads();
    }

    const int64_t out0 = (cur.t * p.Hq + int64_t(cur.kh) * G + og) * D + od;
    if (cur.nsplit == 1) {
      if (has_out) {
#pragma unroll
        for (int e = 0; e < C::OPT; ++e) p.o[out0 + e] = f_bf16(__fdiv_rn(acc[e], l));
      }
    } else {
      const int64_t slot0 = (cur.t * p.Hkv + cur.kh) * int64_t(p.max_splits);
      const int64_t slot = slot0 + cur.s;
      if (has_out) {
#pragma unroll
        for (int e = 0; e < C::OPT; ++e) p.part[(slot * G + og) * D + od + e] = acc[e];
        if (od == 0) {
          p.ml[(slot * G + og) * 2 + 0] =
              fmaxf(fmaxf(red[og * 4 + 0], red[og * 4 + 1]), fmaxf(red[og * 4 + 2], red[og * 4 + 3]));
          p.ml[(slot * G + og) * 2 + 1] = l;
        }
      }
      // Hand-off: the block's stores are ordered before the count by the barrier and the
      // counting thread's GPU-scope fence; the block that counts last merges.
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(p.cnt + cur.t * p.Hkv + cur.kh, 1u);
        s_last = old == uint32_t(cur.nsplit - 1) ? 1u : 0u;
        if (s_last) __threadfence();
      }
      __syncthreads();
      if (s_last && has_out) {
        float M = -INFINITY;
        for (int ss = 0; ss < cur.nsplit; ++ss) M = fmaxf(M, __ldcg(p.ml + ((slot0 + ss) * G + og) * 2));
        float L = 0.0f, A[C::OPT];
#pragma unroll
        for (int e = 0; e < C::OPT; ++e) A[e] = 0.0f;
        for (int ss = 0; ss < cur.nsplit; ++ss) {
          const float f = exp2f(__fsub_rn(__ldcg(p.ml + ((slot0 + ss) * G + og) * 2), M));
          L = __fadd_rn(L, __fmul_rn(__ldcg(p.ml + ((slot0 + ss) * G + og) * 2 + 1), f));
#pragma unroll
          for (int e = 0; e < C::OPT; ++e)
            A[e] = __fadd_rn(A[e], __fmul_rn(__ldcg(p.part + ((slot0 + ss) * G + og) * D + od + e), f));
        }
#pragma unroll
        for (int e = 0; e < C::OPT; ++e) p.o[out0 + e] = f_bf16(__fdiv_rn(A[e], L));
      }
    }
    if (!has_next) break;
    __syncthreads();   // qs and the score buffers are reused by the next unit
    store_q(qn);
    cur = nxt;
    u = un;
    half ^= 1;
  }
  if (bad_page) atomicOr(p.status, kErrPage);
}

struct KernelInfo {
  const void* fn = nullptr;
  size_t (*smem)(int, int) = nullptr;
};

template <int D, int G>
KernelInfo info() {
  KernelInfo k;
  k.fn = reinterpret_cast<const void*>(&attn_kernel<D, G>);
  k.smem = &Cfg<D, G>::smem_bytes;
  return k;
}

inline KernelInfo select(int D, int G) {
  if (D == 128) {
    switch (G) {
      case 1: return info<128, 1>();
      case 2: return info<128, 2>();
      case 4: return info<128, 4>();
      case 8: return info<128, 8>();
    }
  } else if (D == 64) {
    switch (G) {
      case 1: return info<64, 1>();
      case 2: return info<64, 2>();
      case 4: return info<64, 4>();
      case 8: return info<64, 8>();
    }
  }
  return KernelInfo{};
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace biattn

struct bi_attention {
  int Hq = 0, Hkv = 0, D = 0, G = 0, page_size = 0, split = 0;
  float scale = 0.0f;
  int device = 0, num_sms = 0, max_ctas = 0;
  size_t smem = 0;
  int pages_per_split = 0;
  biattn::KernelInfo kern;
  uint32_t* d_status = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

namespace {

struct WsLayout {
  size_t cum, umap, cnt, part, ml, total;
};

WsLayout layout_of(const bi_attention* h, int64_t T, int64_t max_pos) {
  const int64_t max_splits = max_pos / h->split + 1;
  const int64_t slots = T * h->Hkv * max_splits;
  WsLayout w;
  w.cum = 0;
  w.umap = biattn::align256(size_t(T + 1) * sizeof(int32_t));
  w.cnt = w.umap + biattn::align256(size_t(slots) * sizeof(int32_t));
  w.part = w.cnt + biattn::align256(size_t(T) * h->Hkv * sizeof(uint32_t));
  w.ml = w.part + biattn::align256(size_t(slots) * h->G * h->D * sizeof(float));
  w.total = w.ml + biattn::align256(size_t(slots) * h->G * 2 * sizeof(float));
  return w;
}

}  // namespace

BI_GEMM_API int bi_attention_create(bi_attention_t* out, int64_t num_q_heads, int64_t num_kv_heads,
                                    int64_t head_dim, int64_t page_size, float scale, int64_t split_size) {
  if (!out) return BI_GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!std::isfinite(scale) || scale <= 0.0f) return BI_GEMM_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || split_size < 0)
    return BI_GEMM_ERR_INVALID_ARG;
  const int64_t split = split_size ? split_size : biattn::kDefaultSplit;
  if (num_q_heads % num_kv_heads != 0 || num_q_heads > 4096 || page_size > (1 << 20) ||
      split % biattn::kThreads != 0 || split > 1024)
    return BI_GEMM_ERR_UNSUPPORTED;
  const int64_t G = num_q_heads / num_kv_heads;
  const biattn::KernelInfo k = biattn::select(int(head_dim), int(G));
  if (!k.fn) return BI_GEMM_ERR_UNSUPPORTED;

  int dev = 0, major = 0, minor = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return BI_GEMM_ERR_UNSUPPORTED;
  // the most pages one split of `split` positions can touch (its start need not be page-aligned)
  const int pages_per_split = int(split / page_size + 2);
  const size_t smem = k.smem(int(split), pages_per_split);
  // The attribute is per kernel, shared by every handle of the same head shape: set the largest
  // any handle of this kernel can need (split 1024, pages of one position).
  const size_t smem_cap = k.smem(1024, 1024 + 2);
  if (smem_cap > 232448) return BI_GEMM_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_cap)) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, biattn::kThreads, smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  bi_attention* h = new (std::nothrow) bi_attention();
  if (!h) return BI_GEMM_ERR_OOM;
  h->Hq = int(num_q_heads);
  h->Hkv = int(num_kv_heads);
  h->D = int(head_dim);
  h->G = int(G);
  h->page_size = int(page_size);
  h->split = int(split);
  h->scale = scale;
  h->device = dev;
  h->num_sms = sms;
  h->max_ctas = per_sm * sms;
  h->smem = smem;
  h->pages_per_split = pages_per_split;
  h->kern = k;
  if (cudaMalloc(&h->d_status, sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(h->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    if (h->d_status) cudaFree(h->d_status);
    delete h;
    return BI_GEMM_ERR_CUDA;
  }
  *out = h;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_attention_workspace_size(bi_attention_t h, int64_t T, int64_t max_pos, uint64_t* bytes) {
  if (!h || !bytes || T < 0 || max_pos < 0) return BI_GEMM_ERR_INVALID_ARG;
  *bytes = T == 0 ? 0 : uint64_t(layout_of(h, T, max_pos).total);
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_attention_run(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                                 const int32_t* q_pos, const void* k_cache, const void* v_cache,
                                 int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                                 int64_t max_pages, int64_t max_pos, void* o, void* stream) {
  if (!h || T < 0 || num_pages < 0 || num_seqs < 0 || max_pages < 0 || max_pos < 0) return BI_GEMM_ERR_INVALID_ARG;
  if (T == 0) return BI_GEMM_OK;
  if (T > (int64_t(1) << 24) || max_pos >= (int64_t(1) << 30) ||
      T * h->Hkv * (max_pos / h->split + 1) >= (int64_t(1) << 31))   // unit indices are int32
    return BI_GEMM_ERR_UNSUPPORTED;
  if (!q || !q_seq || !q_pos || !k_cache || !v_cache || !page_table || !o) return BI_GEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return BI_GEMM_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(q_seq) | reinterpret_cast<uintptr_t>(q_pos) |
       reinterpret_cast<uintptr_t>(page_table)) & 3u)
    return BI_GEMM_ERR_ALIGNMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (dev != h->device) return BI_GEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsLayout w = layout_of(h, T, max_pos);
  if (w.total > h->ws_bytes) {
    if (h->ws) cudaFreeAsync(h->ws, st);
    h->ws = nullptr;
    h->ws_bytes = 0;
    void* p = nullptr;
    if (cudaMallocAsync(&p, w.total, st) != cudaSuccess) {
      cudaGetLastError();
      return BI_GEMM_ERR_OOM;
    }
    h->ws = p;
    h->ws_bytes = w.total;
  }
  uint8_t* ws = static_cast<uint8_t*>(h->ws);
  biattn::Params p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.q_seq = q_seq;
  p.q_pos = q_pos;
  p.kc = static_cast<const uint16_t*>(k_cache);
  p.vc = static_cast<const uint16_t*>(v_cache);
  p.table = page_table;
  p.o = static_cast<uint16_t*>(o);
  p.cum = reinterpret_cast<int32_t*>(ws + w.cum);
  p.umap = reinterpret_cast<int32_t*>(ws + w.umap);
  p.cnt = reinterpret_cast<uint32_t*>(ws + w.cnt);
  p.part = reinterpret_cast<float*>(ws + w.part);
  p.ml = reinterpret_cast<float*>(ws + w.ml);
  p.status = h->d_status;
  p.T = T;
  p.num_pages = num_pages;
  p.B = num_seqs;
  p.max_pages = max_pages;
  p.Hq = h->Hq;
  p.Hkv = h->Hkv;
  p.page_size = h->page_size;
  p.split = h->split;
  p.max_splits = int32_t(max_pos / h->split + 1);
  p.pages_per_split = h->pages_per_split;
  p.c = h->scale * 1.4426950408889634f;   // log2(e)
  biattn::plan_kernel<<<1, 1024, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return BI_GEMM_ERR_CUDA;
  const int64_t units = T * h->Hkv * int64_t(p.max_splits);
  const unsigned grid = unsigned(std::min<int64_t>(units, h->max_ctas));
  void* args[1] = {&p};
  if (cudaLaunchKernel(h->kern.fn, dim3(grid), dim3(biattn::kThreads), args, h->smem, st) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_attention_get_device_error(bi_attention_t h, void* stream) {
  if (!h) return BI_GEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t s = 0;
  if (cudaMemcpyAsync(&s, h->d_status, sizeof(s), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (s == 0) return BI_GEMM_OK;
  if (cudaMemsetAsync(h->d_status, 0, sizeof(uint32_t), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  return BI_GEMM_ERR_INVALID_ARG;
}

BI_GEMM_API int bi_attention_get_config(bi_attention_t h, bi_attention_config* c) {
  if (!h || !c) return BI_GEMM_ERR_INVALID_ARG;
  c->num_q_heads = h->Hq;
  c->num_kv_heads = h->Hkv;
  c->head_dim = h->D;
  c->page_size = h->page_size;
  c->split_size = h->split;
  c->threads = biattn::kThreads;
  c->stage_positions = biattn::kThreads;
  c->max_ctas = h->max_ctas;
  c->num_sms = h->num_sms;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_attention_destroy(bi_attention_t h) {
  if (!h) return BI_GEMM_OK;
  if (h->ws) cudaFree(h->ws);
  if (h->d_status) cudaFree(h->d_status);
  delete h;
  return BI_GEMM_OK;
}
