// bi_attention.cu — batch-invariant decode attention over a paged KV cache, sm_103a.
// Implements include/bi_attention.h.
//
// "Batch-invariant attention" (nondeterminism article): split the keys of a query at a fixed
// split SIZE, reduce each split in one fixed order, merge the splits in a fixed order.  The
// work unit is (query token t, KV head kh, split s); one block of 128 threads runs a unit:
//   1. the G query heads of kh are held in registers as MMA B fragments (one column per head);
//   2. the split's keys, then its values, stream through a 2-deep ring of 64-position stages
//      (cp.async, 16-byte chunks, row-XOR swizzle so that the ldmatrix reads of both passes are
//      free of bank conflicts); rows past p, or of an invalid page, are zero-filled and masked;
//   3. pass 1: the 64 x G scores of a key stage, S^T = K Q^T on the tensor cores (mma.sync
//      m16n8k16, bf16 in, fp32 accumulate; 16 key positions on the instruction's rows, the G <= 8
//      heads on its columns, each warp 16 positions, k in ascending order), times scale * log2(e);
//   4. per head, the split's maximum m (exact, order-free), the weights w_j = exp2(s_j - m) and
//      their sum l (each thread its positions in order, then a fixed butterfly and warp order);
//   5. pass 2: O^T += V^T P^T on the tensor cores (16 output dimensions on the rows, the heads on
//      the columns), 16 positions per step in ascending order, each warp a quarter of the
//      dimensions; the fp32 weights enter as two bf16 parts (hi = bf16(w), lo = bf16(w - hi), two
//      MMAs), so the products carry 16 of the weights' bits, not 8;
//   6. a single-split token writes bf16(acc / l); otherwise the unit stores (m, l, acc), and a
//      merge kernel combines the n splits of each (token, KV head): M = max m_s, then
//      L = sum l_s 2^(m_s - M) and A = sum acc_s 2^(m_s - M) over four consecutive groups of
//      splits (ascending within a group, the four group sums added in order), o = A / L.
// A plan kernel first turns q_pos into per-token unit offsets (a prefix sum) and a record of
// every unit.  The attention kernel is persistent: a block fetches its next unit's coordinates,
// row offsets and query while it works on the current one and issues the next unit's first
// stages into the ring during the current unit's last ones, so that the key/value stream does
// not drain between units; with the merge in a kernel of its own a unit ends without any fence
// or counter.  For page sizes 8, 16, 32 and 64 a second attention kernel (attn_tma_kernel, below)
// runs the same arithmetic with the keys and values loaded as TMA page boxes by a producer warp.
// The attention and merge kernels are programmatic dependents of their predecessors.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/bi_attention.h"
#include "ptx.cuh"

#ifndef BI_GEMM_API
#define BI_GEMM_API extern "C" __attribute__((visibility("default")))
#endif

namespace biattn {

namespace ptx = bigemm::ptx;

// 3-D tiled bulk tensor load global -> shared (c0 innermost), completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Barrier 1 for kThreadsInBarrier threads (whole warps): synchronises a subset of the block.
template <int kThreadsInBarrier>
__device__ __forceinline__ void named_bar_sync1() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreadsInBarrier) : "memory");
}

// Barrier 1 for kThreadsInBarrier threads with an OR over their predicates: every participant
// gets the same answer.
template <int kThreadsInBarrier>
__device__ __forceinline__ bool named_bar_or1(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(pred)), "n"(kThreadsInBarrier)
      : "memory");
  return r != 0;
}

constexpr int kThreads = 128;        // threads per block (four warps)
constexpr int kStagePos = 64;        // positions per staged key / value tile
constexpr int kMergeThreads = 256;   // merge block: four lanes per output pair, 64 pairs
constexpr int kStages = 2;           // staging ring depth (more blocks per SM beat a deeper ring)
constexpr int kDefaultSplit = 512;
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
  int4* urec;        // [units] (token, request, position, split * Hkv + KV head) of each unit
  float* part;       // [T * Hkv * max_splits, G, D] partial weighted sums
  float* ml;         // [T * Hkv * max_splits, G, 2] (maximum, sum of weights)
  uint32_t* status;
  int64_t T, num_pages, B, max_pages;
  int32_t Hq, Hkv, page_size, split, max_splits;
  int32_t max_pos;   // the host's bound on q_pos
  int32_t nstage;    // ring depth of the TMA variant
  int32_t stall_block;   // failure injection (test controls only): this block never issues its
                         // first load; -1 in the product
  int32_t inline_plan;   // T <= kInlinePlanMaxT: the attention kernel derives unit records itself
  uint64_t timeout_ns;   // limit of its bounded waits
  float c;           // scale * log2(e)
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }


// Number of splits of a token at position p.
__device__ __forceinline__ int32_t splits_of(int32_t p, int32_t split) { return p / split + 1; }

// Unit offsets: cum[t] = Hkv * (splits of the tokens before t), and the record of every unit
// (its token, request, position and split * Hkv + KV head); a token with an input the kernel
// cannot serve gets no units (and sets the status word).
__global__ void __launch_bounds__(1024) plan_kernel(const Params p) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  ptx::launch_dependents();   // the attention kernel may start its prologue now
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < p.T; base += 1024) {
    const int64_t t = base + tid;
    int32_t n = 0, b = 0, pos = 0;
    if (t < p.T) {
      b = p.q_seq[t];
      pos = p.q_pos[t];
      if (b < 0 || b >= p.B || pos < 0 || int64_t(pos / p.page_size) >= p.max_pages) {
        atomicOr(p.status, kErrInput);
      } else if (pos > p.max_pos) {
        atomicOr(p.status, kErrBound);
      } else {
        n = splits_of(pos, p.split) * p.Hkv;
      }
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
    if (t < p.T) p.cum[t] = incl - n;
    // the unit records of the warp's 32 tokens, one token at a time by the whole warp (a long
    // context has hundreds of units)
    for (int k = 0; k < 32; ++k) {
      const int32_t nk = __shfl_sync(0xFFFFFFFFu, n, k);
      const int32_t sk = __shfl_sync(0xFFFFFFFFu, incl - n, k);
      const int32_t bk = __shfl_sync(0xFFFFFFFFu, b, k), pk = __shfl_sync(0xFFFFFFFFu, pos, k);
      const int32_t tk = int32_t(base + warp * 32 + k);
      for (int32_t r = lane; r < nk; r += 32) p.urec[sk + r] = make_int4(tk, bk, pk, r);
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
  static constexpr int STAGE_BYTES = kStagePos * ROW_BYTES;
  static constexpr int CHUNKS_PER_THREAD = kStagePos * CHUNKS / kThreads;
  static constexpr int WPOS = kStagePos / 4;           // positions of a stage per warp (one m tile)
  static constexpr int QS = D + 8;                     // query row stride in shared memory
  static constexpr int KSTEPS = D / 16;                // k steps of the score MMA
  static constexpr int DW = D / 4;                     // output dimensions per warp
  static constexpr int MT2 = DW / 16;                  // m tiles (16 dimensions) per warp in the value MMA
  static_assert(G <= 8, "the query heads of a group fill at most the MMA's 8 columns");
  static_assert(WPOS == 16 && MT2 >= 1 && DW % 16 == 0, "warp layout: 16 positions, 16-dimension tiles");
  // score row stride (floats): a multiple of 8 keeps float2 rows aligned; +8 spreads the banks
  __host__ __device__ static int sc_stride(int split) { return split + 8; }
  // ring | row offsets [2][split] (int64) | scores [G][stride] | per-warp maxima [G][4] |
  // per-warp sums [G][4] | maximum [G] | sum [G] | query rows [2][G][QS] (bf16)
  static size_t smem_bytes(int split) {
    return size_t(kStages) * STAGE_BYTES + sizeof(int64_t) * 2 * size_t(split) +
           sizeof(float) * (size_t(G) * sc_stride(split) + G * 10) + sizeof(uint16_t) * 2 * G * QS;
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

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

// d += a * b on the tensor cores: a 16 x 16 (row-major, bf16), b 16 x 8 (column-major, bf16),
// d 16 x 8 fp32.  Both passes put the G <= 8 query heads of a unit on the 8 columns (n) and 16
// positions (scores) or 16 output dimensions (values) on the rows (m), so that every row of the
// instruction carries data:
//   scores  S^T = K Q^T:  a = 16 key rows x 16 dimensions, b = the query rows (column = head);
//   values  O^T += V^T P^T:  a = 16 dimensions x 16 value rows, b = the weights (column = head).
// Fragment coordinates (gq = lane / 4, tq = lane % 4): a0 = a[gq][2tq, +1], a1 = a[gq + 8][2tq, +1],
// a2 = a[gq][2tq + 8, +1], a3 = a[gq + 8][2tq + 8, +1]; b0 = b[2tq, +1][gq], b1 = b[2tq + 8, +1][gq];
// d0, d1 = d[gq][2tq, +1], d2, d3 = d[gq + 8][2tq, +1].
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One unit's coordinates, read from the plan.
struct Unit {
  int64_t t, b;
  int32_t kh, s, pos, nsplit, j0, valid, nsub;
};

__device__ __forceinline__ Unit unit_from(const Params& p, const int4 rec) {
  Unit w;
  w.t = rec.x;
  w.b = rec.y;
  w.pos = rec.z;
  w.s = rec.w / p.Hkv;
  w.kh = rec.w - w.s * p.Hkv;
  w.nsplit = splits_of(w.pos, p.split);
  w.j0 = w.s * p.split;
  w.valid = min(p.split, w.pos + 1 - w.j0);                  // keys in this split (>= 1)
  w.nsub = (w.valid + kStagePos - 1) / kStagePos;
  return w;
}

// Small batches (T <= kInlinePlanMaxT tokens) skip the plan kernel: a warp derives a unit's
// record from q_seq / q_pos itself, with the plan's numbering (tokens in order, a token's units
// numbered split * Hkv + KV head, no units for a token the kernel cannot serve).  The tokens are
// loaded first (plan_load) and scanned later (plan_find), so that the load latency
// can overlap other work.
constexpr int kInlinePlanMaxT = 32;

struct PlanRegs {
  int32_t b[kInlinePlanMaxT / 32 + 1], pos[kInlinePlanMaxT / 32 + 1];
};

__device__ __forceinline__ void plan_load(const Params& p, PlanRegs& r) {
  const int lane = int(threadIdx.x) & 31;
#pragma unroll
  for (int k = 0; k < kInlinePlanMaxT / 32 + 1; ++k) {
    const int64_t t = int64_t(k * 32 + lane);
    r.b[k] = t < p.T ? p.q_seq[t] : -1;
    r.pos[k] = t < p.T ? p.q_pos[t] : -1;
  }
}

// Warp-collective (all 32 lanes): the record of unit u (x = -1 when u is past the last unit) and
// the total number of units.  With `report`, tokens the kernel cannot serve set the status word.
__device__ __forceinline__ int4 plan_find(const Params& p, const PlanRegs& r, int64_t u, int32_t* total,
                                          bool report) {
  const int lane = int(threadIdx.x) & 31;
  int32_t carry = 0;
  int4 rec = make_int4(-1, 0, 0, 0);
#pragma unroll
  for (int k = 0; k < kInlinePlanMaxT / 32 + 1; ++k) {
    const int64_t t = int64_t(k * 32 + lane);
    const int32_t b = r.b[k], pos = r.pos[k];
    int32_t n = 0;
    if (t < p.T) {
      if (b < 0 || b >= p.B || pos < 0 || int64_t(pos / p.page_size) >= p.max_pages) {
        if (report) atomicOr(p.status, kErrInput);
      } else if (pos > p.max_pos) {
        if (report) atomicOr(p.status, kErrBound);
      } else {
        n = splits_of(pos, p.split) * p.Hkv;
      }
    }
    int32_t x = n;   // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    const int32_t ex = carry + x - n;
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, n > 0 && u >= ex && u < int64_t(ex) + n);
    if (hit) {
      const int src = __ffs(int(hit)) - 1;
      const int32_t e = __shfl_sync(0xFFFFFFFFu, ex, src);
      rec = make_int4(k * 32 + src, __shfl_sync(0xFFFFFFFFu, b, src), __shfl_sync(0xFFFFFFFFu, pos, src),
                      int32_t(u - e));
    }
    carry += __shfl_sync(0xFFFFFFFFu, x, 31);
  }
  *total = carry;
  return rec;
}

// A unit's outputs from the value accumulators of one warp (acc[mt][e]: head 2tq + (e & 1),
// dimension dbase + 16mt + gq + 8(e >> 1)): o = bf16(acc / l) for a single-split token, or the
// fp32 partial sums of the split.
template <int D, int G, int MT2>
__device__ __forceinline__ void store_out(const Params& p, const Unit& w, const float (&acc)[MT2][4],
                                          const float* hl, int dbase, int lane) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int h = 2 * tq + (e & 1);
    if (h < G) {
      const float l = hl[h];
      uint16_t* orow = p.o + (w.t * p.Hq + int64_t(w.kh) * G + h) * D + dbase + gq + (e >> 1) * 8;
#pragma unroll
      for (int mt = 0; mt < MT2; ++mt) orow[16 * mt] = uint16_t(pack_bf16x2(__fdiv_rn(acc[mt][e], l), 0.0f));
    }
  }
}

template <int D, int G, int MT2>
__device__ __forceinline__ void store_partial(const Params& p, int64_t slot, const float (&acc)[MT2][4], int dbase,
                                              int lane) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int h = 2 * tq + (e & 1);
    if (h < G) {
      float* prow = p.part + (slot * G + h) * D + dbase + gq + (e >> 1) * 8;
#pragma unroll
      for (int mt = 0; mt < MT2; ++mt) prow[16 * mt] = acc[mt][e];
    }
  }
}

template <int D, int G, bool kInline>
__global__ void __launch_bounds__(kThreads, 4) attn_kernel(const Params p) {
  using C = Cfg<D, G>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  const int SCS = C::sc_stride(p.split);
  int64_t* rowoff = reinterpret_cast<int64_t*>(smem + kStages * C::STAGE_BYTES);   // [2][split]
  float* sc = reinterpret_cast<float*>(rowoff + 2 * p.split);               // [G][SCS] scores, then weights
  float* red = sc + G * SCS;                                                // [G][4] per-warp maxima
  float* redl = red + G * 4;                                                // [G][4] per-warp sums
  float* hm = redl + G * 4;                                                 // [G] maximum of the split
  float* hl = hm + G;                                                       // [G] sum of its weights
  uint16_t* qsm = reinterpret_cast<uint16_t*>(hl + G);                      // [2][G][D + 8] query rows
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;       // MMA fragment coordinates: row (head), pair
  const bool row_ok = gq < G;
  const int dbase = warp * C::DW;               // this warp's output dimensions

  ptx::grid_dependency_wait();   // the plan (or the previous kernel) is complete and visible
  ptx::launch_dependents();
  int64_t u = blockIdx.x;
  int32_t total = 0;
  int4 rec0 = make_int4(0, 0, 0, 0);
  if constexpr (kInline) {
    PlanRegs pr;
    plan_load(p, pr);
    rec0 = plan_find(p, pr, u, &total, blockIdx.x == 0 && tid < 32);
  } else {
    total = p.cum[p.T];
    if (u < total) rec0 = p.urec[u];
  }
  if (u >= total) return;
  // record of a later unit of this block
  auto record = [&](int64_t w) {
    if constexpr (!kInline) {
      return p.urec[w];
    } else {
      PlanRegs pr;
      int32_t tot;
      plan_load(p, pr);
      return plan_find(p, pr, w, &tot, false);
    }
  };

  // Element offset of each key / value row of a unit's split in the caches (without the KV head),
  // or -1 for a row whose page index is outside [0, num_pages).
  auto fill_rows = [&](const Unit& w, int half) {
    for (int jl = tid; jl < w.valid; jl += kThreads) {
      const int32_t j = w.j0 + jl;
      const int64_t page = p.table[w.b * p.max_pages + j / p.page_size];
      rowoff[half * p.split + jl] =
          (page >= 0 && page < p.num_pages) ? (page * p.page_size + j % p.page_size) * p.Hkv * D : int64_t(-1);
    }
  };
  // A unit's G query rows go to its half of qsm (rows padded by 8 elements, so that the
  // fragment reads of the eight heads fall in different banks).
  auto load_q = [&](const Unit& w, int half) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q + (w.t * p.Hq + int64_t(w.kh) * G) * D);
    uint32_t* dst = reinterpret_cast<uint32_t*>(qsm + half * G * C::QS);
    for (int i = tid; i < G * D / 2; i += kThreads) dst[(i / (D / 2)) * (C::QS / 2) + i % (D / 2)] = src[i];
  };

  bool bad_page = false;
  // Load number i of unit w (key stages, then value stages) into ring slot `slot`.
  auto issue = [&](const Unit& w, int half, int i, int slot) {
    const bool isv = i >= w.nsub;
    const int sub = isv ? i - w.nsub : i;
    const uint16_t* base = isv ? p.vc : p.kc;
    const uint32_t dst0 = ptx::smem_u32(ring + slot * C::STAGE_BYTES);
    const int64_t* ro = rowoff + half * p.split + sub * kStagePos;
    const uint16_t* hbase = base + int64_t(w.kh) * D;
    const int rows = w.valid - sub * kStagePos;
#pragma unroll 4
    for (int it = 0; it < C::CHUNKS_PER_THREAD; ++it) {
      const int lin = it * kThreads + tid;
      const int row = lin / C::CHUNKS, c = lin % C::CHUNKS;
      const uint32_t dst = dst0 + row * C::ROW_BYTES + ((c ^ (row & (C::CHUNKS - 1))) << 4);
      const void* src = base;
      uint32_t bytes = 0;
      if (row < rows) {
        const int64_t off = ro[row];
        if (off >= 0) {
          src = hbase + off + c * 8;
          bytes = 16;
        } else {
          bad_page = true;
        }
      }
      ptx::cp_async_16(dst, src, bytes);   // bytes == 0: zero-fill, nothing read
    }
  };
  // Shared-memory address of 16-byte chunk c of staged row r.
  auto chunk_addr = [&](uint32_t stage, int r, int c) {
    return stage + r * C::ROW_BYTES + ((c ^ (r & (C::CHUNKS - 1))) << 4);
  };

  Unit cur = unit_from(p, rec0);
  int half = 0;
  load_q(cur, half);
  fill_rows(cur, half);
  __syncthreads();
  uint32_t seq = 0;   // sequence number of the next load to issue (its ring slot is seq % kStages)
  uint32_t cons = 0;  // sequence number of the next load to consume
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < 2 * cur.nsub) issue(cur, half, i, int(seq % kStages));
    ++seq;
    ptx::cp_async_commit();
  }

  while (true) {
    // The next unit of this block: its coordinates, row offsets and query are fetched while this
    // unit's first stage is awaited (or up front when this unit has a single key stage, since
    // the next unit's first load is then issued right away), so that its first stages can be
    // issued during this unit's last ones.
    const int64_t un = u + gridDim.x;
    const bool has_next = un < total;
    Unit nxt;
    auto fetch_next = [&]() {
      if (has_next) {
        nxt = unit_from(p, record(un));
        fill_rows(nxt, half ^ 1);
        load_q(nxt, half ^ 1);
      }
    };
    const int nload = 2 * cur.nsub;
    if (nload <= kStages - 1) {
      fetch_next();
      __syncthreads();   // the next unit's row offsets are visible to every issuing thread
    }
    float acc[C::MT2][4];
#pragma unroll
    for (int n = 0; n < C::MT2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
    for (int i = 0; i < nload; ++i) {
      const int ahead = i + kStages - 1;   // the load issued now: this unit's, or the next's
      if (ahead < nload) issue(cur, half, ahead, int(seq % kStages));
      else if (has_next && ahead - nload < 2 * nxt.nsub) issue(nxt, half ^ 1, ahead - nload, int(seq % kStages));
      ++seq;
      ptx::cp_async_commit();
      if (i == 0 && nload > kStages - 1) fetch_next();   // visible after the barrier below
      ptx::cp_async_wait<kStages - 1>();
      __syncthreads();
      const uint32_t stage = ptx::smem_u32(ring + (cons % kStages) * C::STAGE_BYTES);
      ++cons;
      if (i < cur.nsub) {
        // pass 1: scores of this warp's 16 positions of the stage, S^T = K Q^T on the tensor
        // cores, fixed k order: rows gq and gq + 8 (positions), columns 2tq and 2tq + 1 (heads)
        const int pos0 = i * kStagePos + warp * C::WPOS;
        // query B fragments: b0 = q[gq][16k + 2tq, +1], b1 = q[gq][16k + 8 + 2tq, +1] (zero past the G heads)
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qsm + (half * G + (row_ok ? gq : 0)) * C::QS);
        // key A fragments: the four 8 x 8 blocks (rows 0-7 | 8-15) x (dimensions 0-7 | 8-15) of the k step
        const int prow = warp * C::WPOS + ((lane >> 3) & 1) * 8 + (lane & 7);
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < C::KSTEPS; ++k) {
          uint32_t a[4];
          ldsm_x4(chunk_addr(stage, prow, 2 * k + (lane >> 4)), a);
          mma16816(d, a, row_ok ? qrow[8 * k + tq] : 0u, row_ok ? qrow[8 * k + 4 + tq] : 0u);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = 2 * tq + (e & 1), jl = pos0 + gq + (e >> 1) * 8;
          if (h < G && jl < cur.valid) sc[h * SCS + jl] = __fmul_rn(d[e], p.c);
        }
        if (i == cur.nsub - 1) {
          // the split's maximum per head, the weights in place and their sum (fixed tree)
          __syncthreads();
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float m = -INFINITY;
            for (int jj = tid; jj < cur.valid; jj += kThreads) m = fmaxf(m, sc[g * SCS + jj]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if (lane == 0) red[g * 4 + warp] = m;
          }
          __syncthreads();
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float m = fmaxf(fmaxf(red[g * 4 + 0], red[g * 4 + 1]), fmaxf(red[g * 4 + 2], red[g * 4 + 3]));
            float ls = 0.0f;
            for (int jj = tid; jj < cur.valid; jj += kThreads) {
              const float w = exp2f(__fsub_rn(sc[g * SCS + jj], m));
              sc[g * SCS + jj] = w;
              ls = __fadd_rn(ls, w);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xFFFFFFFFu, ls, o));
            if (tid == 0) hm[g] = m;
            if (lane == 0) redl[g * 4 + warp] = ls;
          }
          __syncthreads();
          if (tid < G)
            hl[tid] = __fadd_rn(__fadd_rn(__fadd_rn(redl[tid * 4 + 0], redl[tid * 4 + 1]), redl[tid * 4 + 2]),
                                redl[tid * 4 + 3]);
        }
      } else {
        // pass 2: O^T += V^T P^T over this stage's positions, 16 at a time, on the tensor cores;
        // P (fp32) enters as two bf16 parts, hi = bf16(P) and lo = bf16(P - hi), each an MMA
        const int sub = i - cur.nsub;
        const int rows = min(kStagePos, cur.valid - sub * kStagePos);
        for (int k0 = 0; k0 < rows; k0 += 16) {
          float pw[4];
          const int jb = sub * kStagePos + k0 + 2 * tq;   // position (within the split) of pw[0]
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int jl = jb + (e >> 1) * 8 + (e & 1);
            pw[e] = (row_ok && jl < cur.valid) ? sc[gq * SCS + jl] : 0.0f;
          }
          uint32_t ah[2], al[2];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const float x0 = pw[2 * h2], x1 = pw[2 * h2 + 1];
            ah[h2] = pack_bf16x2(x0, x1);
            const float h0 = __uint_as_float(ah[h2] << 16), h1 = __uint_as_float(ah[h2] & 0xFFFF0000u);
            al[h2] = pack_bf16x2(__fsub_rn(x0, h0), __fsub_rn(x1, h1));
          }
          // value A fragments (transposed loads): the blocks (positions 0-7 | 8-15) x
          // (dimensions 0-7 | 8-15) of the m tile; the weights are the B fragments
#pragma unroll
          for (int mt = 0; mt < C::MT2; ++mt) {
            uint32_t a[4];
            const int prow = k0 + (lane >> 4) * 8 + (lane & 7);
            ldsm_x4_trans(chunk_addr(stage, prow, (dbase + 16 * mt) / 8 + ((lane >> 3) & 1)), a);
            mma16816(acc[mt], a, ah[0], ah[1]);
            mma16816(acc[mt], a, al[0], al[1]);
          }
        }
      }
      __syncthreads();
    }

    // this thread's outputs: heads 2tq and 2tq + 1, dimensions dbase + 16mt + gq and + 8 of
    // each m tile
    if (cur.nsplit == 1) {
      store_out<D, G>(p, cur, acc, hl, dbase, lane);
    } else {
      const int64_t slot0 = (cur.t * p.Hkv + cur.kh) * int64_t(p.max_splits);
      const int64_t slot = slot0 + cur.s;
      store_partial<D, G>(p, slot, acc, dbase, lane);
      if (tid < G) {
        p.ml[(slot * G + tid) * 2 + 0] = hm[tid];
        p.ml[(slot * G + tid) * 2 + 1] = hl[tid];
      }
    }
    if (!has_next) break;
    __syncthreads();   // scores and per-head values are reused by the next unit
    cur = nxt;
    u = un;
    half ^= 1;
  }
  if (bad_page) atomicOr(p.status, kErrPage);
}

// ------------------------------------------------------------------ TMA page-box variant
// The same unit arithmetic for page sizes 8, 16, 32 and 64, where a 64-position stage is whole
// pages.  Warp 0 is a producer: for every page of a stage it loads the rows of the unit's KV
// head as [page_size x 64] boxes (two per page for a head dimension of 128) with 3-D TMA,
// 128-byte swizzled, into a ring of stages and runs ahead across units; a page index outside
// the cache loads a box from past the cache's end, which TMA fills with zeros (the rows the
// row-copy kernel zero-fills).  Warps 1..4 compute exactly as attn_kernel's four warps do (same
// instructions in the same order on the same values), so both kernels give the same bits.  Both
// roles read the next unit's record one unit ahead (the producer also its page-table entries,
// the consumers its query rows), so that no dependent load stalls the stream at a unit change.
// Every wait on the ring is bounded: past the limit the block sets kErrTimeout, stops issuing,
// waits (bounded) for the copies it has in flight, and leaves.
// Four consumer warps per block, each with the share of a stage (16 positions) and of the output
// (D / 4 dimensions) that the same warp of attn_kernel has, so that every score and every output
// element goes through the same instructions in the same order.  (Eight consumer warps at two
// blocks per SM were measured slower than four at three.)
constexpr int kTmaConsumerWarps = 4;
constexpr int kTmaBlocksPerSm = 3;   // the ring of the default build is sized for these
constexpr int kTmaMaxStages = 8;
constexpr uint32_t kErrTimeout = 8u;          // a bounded wait on the ring expired
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D, int G>
struct TmaCfg {
  using C = Cfg<D, G>;
  static constexpr int CW = kTmaConsumerWarps;
  static constexpr int CT = 32 * CW;                   // consumer threads
  static constexpr int THREADS = 32 + CT;              // producer warp + consumers
  static constexpr int BLOCKS_PER_SM = kTmaBlocksPerSm;
  static_assert(CW == 4 && C::WPOS * CW == kStagePos, "consumer warp layout: attn_kernel's");
  static constexpr int HALVES = D / 64;                // 128-byte column halves of a row
  static constexpr int HALF_BYTES = kStagePos * 128;   // one half of a stage: 64 rows of 128 B
  static constexpr int STAGE_BYTES = HALVES * HALF_BYTES;
  static constexpr int QW = (G * D / 2 + CT - 1) / CT;   // query words per consumer
  // 1024-byte alignment slack | ring [nstage] | full, empty barriers [nstage] each | scores
  // [G][stride] | per-warp maxima, sums [G][4] each | maximum, sum [G] each | query rows [G][QS]
  // (the host adds nstage x (STAGE_BYTES + 16) for the ring and its barriers)
  static size_t fixed_bytes(int split) {
    return 1024 + sizeof(float) * (size_t(G) * C::sc_stride(split) + G * 10) + sizeof(uint16_t) * G * C::QS;
  }
};

// Bounded wait for a phase of a ring barrier: false (status set, block aborted) past the time
// limit, or at once once another role of the block has aborted.
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, const Params& p, volatile uint32_t* abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (ptx::globaltimer() - t0 > p.timeout_ns) {
      atomicOr(p.status, kErrTimeout);
      *abort = 1u;
      return false;
    }
  }
  return true;
}

// kBlocksPerSm: the resident blocks per SM the registers are budgeted for: 3, with the ring sized
// for them, or 4, with the ring that four blocks leave room for (two stages at a head dimension of
// 128), so that a call of up to four units per SM runs in one round.
template <int D, int G, bool kInline, int kBlocksPerSm>
__global__ void __launch_bounds__(TmaCfg<D, G>::THREADS, kBlocksPerSm)
    attn_tma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const Params p) {
  using C = Cfg<D, G>;
  using TC = TmaCfg<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int NS = p.nstage;
  const int SCS = C::sc_stride(p.split);
  const uint32_t bars = sbase + uint32_t(NS * TC::STAGE_BYTES);   // full [NS], then empty [NS]
  float* sc = reinterpret_cast<float*>(smem + NS * TC::STAGE_BYTES + 16 * NS);   // [G][SCS]
  float* red = sc + G * SCS;
  float* redl = red + G * 4;
  float* hm = redl + G * 4;
  float* hl = hm + G;
  uint16_t* qsm = reinterpret_cast<uint16_t*>(hl + G);   // [G][QS]
  __shared__ uint32_t s_abort;
  volatile uint32_t* abort = &s_abort;
  const int tid = int(threadIdx.x), lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_abort = 0u;
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(bars + 8 * s, 1);
      ptx::mbar_init(bars + 8 * (NS + s), TC::CW);
    }
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&tmk);
    ptx::prefetch_tensormap(&tmv);
  }
  __syncthreads();
  ptx::grid_dependency_wait();   // the plan (or the previous kernel) is complete and visible
  ptx::launch_dependents();
  int32_t total = 0;
  int4 rec0 = make_int4(0, 0, 0, 0);
  if constexpr (kInline) {
    PlanRegs pr;
    plan_load(p, pr);
    rec0 = plan_find(p, pr, int64_t(blockIdx.x), &total, blockIdx.x == 0 && warp == 0);
  } else {
    total = p.cum[p.T];
    if (int64_t(blockIdx.x) < total) rec0 = p.urec[blockIdx.x];
  }
  if (int64_t(blockIdx.x) >= total) return;
  // The next unit's record is fetched in two steps a stage apart: the plan's table entry, or
  // with the inline plan the tokens' positions (first step) and the warp's scan (second step).
  PlanRegs npr;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int ps = p.page_size;
    const int ppst = kStagePos / ps;                   // pages per stage: 1, 2, 4 or 8
    const uint32_t box_bytes = uint32_t(ps) * 128;
    const int32_t past_end = int32_t(p.num_pages * ps);   // a row coordinate past the cache
    // page-table entries of a unit: lane l holds those of its pages l, l + 32, l + 64, l + 96
    auto load_pages = [&](const Unit& w, int32_t (&pg)[4]) {
      const int npu = (w.valid + ps - 1) / ps;
      const int32_t* row = p.table + w.b * p.max_pages + w.j0 / ps;
#pragma unroll
      for (int k = 0; k < 4; ++k) pg[k] = lane + 32 * k < npu ? row[lane + 32 * k] : -1;
    };
    bool bad_page = false, stop = false;
    uint32_t seq = 0;   // loads issued
    int64_t u = blockIdx.x;
    Unit cur = unit_from(p, rec0);
    int32_t pg[4];
    load_pages(cur, pg);
    while (!stop) {
      const int64_t un = u + gridDim.x;
      const bool has_next = un < total;
      int4 nrec = make_int4(0, 0, 0, 0);
      Unit nxt = cur;
      int32_t npg[4] = {-1, -1, -1, -1};
      const int nload = 2 * cur.nsub;
      const int npu = (cur.valid + ps - 1) / ps;
      for (int i = 0; i < nload; ++i, ++seq) {
        if (i == 0 && has_next) {
          if constexpr (kInline) plan_load(p, npr);
          else nrec = p.urec[un];
        }
        if (i == 1 && has_next) {
          if constexpr (kInline) {
            int32_t tot;
            nrec = plan_find(p, npr, un, &tot, false);
          }
          nxt = unit_from(p, nrec);
          load_pages(nxt, npg);
        }
        const int slot = int(seq % uint32_t(NS));
        const uint32_t round = seq / uint32_t(NS);
        bool ok = true;
        if (lane == 0 && round > 0) ok = ring_wait(bars + 8 * (NS + slot), (round - 1) & 1u, p, abort);
        if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) {
          stop = true;
          break;
        }
        const bool isv = i >= cur.nsub;
        const int sub = isv ? i - cur.nsub : i;
        const int idx0 = sub * ppst;                     // first page of the stage in the unit
        const int cnt = min(ppst, npu - idx0);           // pages of the stage that hold keys
        const uint32_t full = bars + 8 * slot;
        if (seq == 0 && int(blockIdx.x) == p.stall_block) continue;
        if (lane == 0) ptx::mbar_arrive_expect_tx(full, uint32_t(cnt * TC::HALVES) * box_bytes);
        __syncwarp();
        const int k = idx0 >> 5, l0 = idx0 & 31;         // a stage's pages sit in one register
        if (lane >= l0 && lane < l0 + cnt) {
          const int32_t page = k == 0 ? pg[0] : k == 1 ? pg[1] : k == 2 ? pg[2] : pg[3];
          int32_t row = past_end;
          if (page >= 0 && int64_t(page) < p.num_pages) row = page * ps;
          else bad_page = true;
          const uint32_t dst = sbase + uint32_t(slot * TC::STAGE_BYTES) + uint32_t(lane - l0) * box_bytes;
#pragma unroll
          for (int hh = 0; hh < TC::HALVES; ++hh)
            tma_load_3d(dst + hh * TC::HALF_BYTES, isv ? &tmv : &tmk, full, hh * 64, cur.kh, row);
        }
      }
      if (stop || !has_next) break;
      cur = nxt;
      u = un;
#pragma unroll
      for (int k = 0; k < 4; ++k) pg[k] = npg[k];
    }
    if (bad_page) atomicOr(p.status, kErrPage);
    // the block must not leave while a copy into its shared memory is in flight: wait (bounded)
    // for the latest load of every slot
    if (lane == 0) {
      for (uint32_t k = 0; k < uint32_t(NS) && k < seq; ++k) {
        const uint32_t q = seq - 1 - k;
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(bars + 8 * (q % uint32_t(NS)), (q / uint32_t(NS)) & 1u)) {
          if (ptx::globaltimer() - t0 > p.timeout_ns) {
            atomicOr(p.status, kErrTimeout);
            break;
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = tid - 32, cw = warp - 1;
  const int gq = lane >> 2, tq = lane & 3;
  const bool row_ok = gq < G;
  const int dbase = cw * C::DW;
  constexpr int CT = TC::CT;
  // 16-byte chunk c of staged row r (the boxes' 128-byte swizzle: two column halves of 64 rows)
  auto chunk_addr = [&](uint32_t stage, int r, int c) {
    return stage + uint32_t((c >> 3) * TC::HALF_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  };
  auto load_q = [&](const Unit& w, uint32_t (&qr)[TC::QW]) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q + (w.t * p.Hq + int64_t(w.kh) * G) * D);
#pragma unroll
    for (int k = 0; k < TC::QW; ++k) {
      const int i = ctid + k * CT;
      qr[k] = i < G * D / 2 ? src[i] : 0u;
    }
  };
  int64_t u = blockIdx.x;
  Unit cur = unit_from(p, rec0);
  uint32_t qr[TC::QW];
  load_q(cur, qr);
  uint32_t seq = 0;
  bool ok = true;   // false once a wait gave up: the warp then skips the work but walks the barriers
  while (true) {
    {
      uint32_t* dst = reinterpret_cast<uint32_t*>(qsm);
#pragma unroll
      for (int k = 0; k < TC::QW; ++k) {
        const int i = ctid + k * CT;
        if (i < G * D / 2) dst[(i / (D / 2)) * (C::QS / 2) + i % (D / 2)] = qr[k];
      }
    }
    named_bar_sync1<CT>();
    // this thread's query A fragments for every k step, held for the unit:
    // qa[k][0] = q[gq][16k + 2tq, +1], qa[k][1] = q[gq][16k + 8 + 2tq, +1] (zero past the G heads)
    uint32_t qa[C::KSTEPS][2];
    {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qsm + (row_ok ? gq : 0) * C::QS);
#pragma unroll
      for (int k = 0; k < C::KSTEPS; ++k) {
        qa[k][0] = row_ok ? qrow[8 * k + tq] : 0u;
        qa[k][1] = row_ok ? qrow[8 * k + 4 + tq] : 0u;
      }
    }
    const int64_t un = u + gridDim.x;
    const bool has_next = un < total;
    int4 nrec = make_int4(0, 0, 0, 0);
    Unit nxt = cur;
    const int nload = 2 * cur.nsub;
    float acc[C::MT2][4];
#pragma unroll
    for (int n = 0; n < C::MT2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
    for (int i = 0; i < nload; ++i, ++seq) {
      if (i == 0 && has_next) {
        if constexpr (kInline) plan_load(p, npr);
        else nrec = p.urec[un];
      }
      if (i == 1 && has_next) {
        if constexpr (kInline) {
          int32_t tot;
          nrec = plan_find(p, npr, un, &tot, false);
        }
        nxt = unit_from(p, nrec);
        load_q(nxt, qr);
      }
      const int slot = int(seq % uint32_t(NS));
      if (ok && !ring_wait(bars + 8 * slot, (seq / uint32_t(NS)) & 1u, p, abort)) ok = false;
      ok = __all_sync(0xFFFFFFFFu, ok);   // the warp's MMAs run with all lanes or none
      const uint32_t stage = sbase + uint32_t(slot * TC::STAGE_BYTES);
      if (i < cur.nsub) {
        if (ok) {
          // S^T = K Q^T for this warp's 16 positions, as in attn_kernel
          const int pos0 = i * kStagePos + cw * C::WPOS;
          const int prow = cw * C::WPOS + ((lane >> 3) & 1) * 8 + (lane & 7);
          float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int k = 0; k < C::KSTEPS; ++k) {
            uint32_t a[4];
            ldsm_x4(chunk_addr(stage, prow, 2 * k + (lane >> 4)), a);
            mma16816(d, a, qa[k][0], qa[k][1]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = 2 * tq + (e & 1), jl = pos0 + gq + (e >> 1) * 8;
            if (h < G && jl < cur.valid) sc[h * SCS + jl] = __fmul_rn(d[e], p.c);
          }
        }
        if (i == cur.nsub - 1) {
          // the split's maximum, weights and sum: attn_kernel's 128-thread tree, on consumer
          // warps 0..3 (the others wait at the barriers)
          named_bar_sync1<CT>();
          if (cw < 4) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float m = -INFINITY;
              for (int jj = ctid; jj < cur.valid; jj += kThreads) m = fmaxf(m, sc[g * SCS + jj]);
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
              if (lane == 0) red[g * 4 + cw] = m;
            }
          }
          named_bar_sync1<CT>();
          if (cw < 4) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float m = fmaxf(fmaxf(red[g * 4 + 0], red[g * 4 + 1]), fmaxf(red[g * 4 + 2], red[g * 4 + 3]));
              float ls = 0.0f;
              for (int jj = ctid; jj < cur.valid; jj += kThreads) {
                const float w = exp2f(__fsub_rn(sc[g * SCS + jj], m));
                sc[g * SCS + jj] = w;
                ls = __fadd_rn(ls, w);
              }
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xFFFFFFFFu, ls, o));
              if (ctid == 0) hm[g] = m;
              if (lane == 0) redl[g * 4 + cw] = ls;
            }
          }
          named_bar_sync1<CT>();
          if (ctid < G)
            hl[ctid] = __fadd_rn(__fadd_rn(__fadd_rn(redl[ctid * 4 + 0], redl[ctid * 4 + 1]), redl[ctid * 4 + 2]),
                                 redl[ctid * 4 + 3]);
        }
      } else {
        const int sub = i - cur.nsub;
        const int rows = min(kStagePos, cur.valid - sub * kStagePos);
        if (rows & 15) {
          // the value rows the last 16-position step reads past the split's keys (another
          // request's slots of a partly used page, or an earlier stage) become zeros: they meet
          // zero weights, as the zero-filled rows of attn_kernel do
          if (ok) {
            const int r0 = rows, nr = ((rows + 15) & ~15) - rows;
            for (int e = ctid; e < nr * (D / 8); e += CT)
              ptx::st_shared_v4(chunk_addr(stage, r0 + e / (D / 8), e % (D / 8)), 0u, 0u, 0u, 0u);
            ptx::fence_proxy_async_smem();   // ordered before the slot's next TMA write
          }
          named_bar_sync1<CT>();
        }
        if (ok) {
          for (int k0 = 0; k0 < rows; k0 += 16) {
            // weights of positions jb, jb + 1, jb + 8, jb + 9 (zero past the split's keys)
            const int jb = sub * kStagePos + k0 + 2 * tq;
            const float* srow = sc + (row_ok ? gq : 0) * SCS;
            const float2 w0 = *reinterpret_cast<const float2*>(srow + jb);
            const float2 w1 = *reinterpret_cast<const float2*>(srow + jb + 8);
            float pw[4] = {w0.x, w0.y, w1.x, w1.y};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (!row_ok || jb + (e >> 1) * 8 + (e & 1) >= cur.valid) pw[e] = 0.0f;
            uint32_t ah[2], al[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const float x0 = pw[2 * h2], x1 = pw[2 * h2 + 1];
              ah[h2] = pack_bf16x2(x0, x1);
              const float h0 = __uint_as_float(ah[h2] << 16), h1 = __uint_as_float(ah[h2] & 0xFFFF0000u);
              al[h2] = pack_bf16x2(__fsub_rn(x0, h0), __fsub_rn(x1, h1));
            }
#pragma unroll
            for (int mt = 0; mt < C::MT2; ++mt) {
              uint32_t a[4];
              const int prow = k0 + (lane >> 4) * 8 + (lane & 7);
              ldsm_x4_trans(chunk_addr(stage, prow, (dbase + 16 * mt) / 8 + ((lane >> 3) & 1)), a);
              mma16816(acc[mt], a, ah[0], ah[1]);
              mma16816(acc[mt], a, al[0], al[1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + 8 * (NS + slot));   // this warp is done with the slot
    }

    named_bar_sync1<CT>();   // hl is written
    if (ok) {
      if (cur.nsplit == 1) {
        store_out<D, G>(p, cur, acc, hl, dbase, lane);
      } else {
        const int64_t slot = (cur.t * p.Hkv + cur.kh) * int64_t(p.max_splits) + cur.s;
        store_partial<D, G>(p, slot, acc, dbase, lane);
        if (ctid < G) {
          p.ml[(slot * G + ctid) * 2 + 0] = hm[ctid];
          p.ml[(slot * G + ctid) * 2 + 1] = hl[ctid];
        }
      }
    }
    // the scores, per-head values and query rows are reused by the next unit; every consumer
    // warp takes the same decision to go on
    if (named_bar_or1<CT>(!ok) || !has_next) break;
    cur = nxt;
    u = un;
  }
}

// Merge of the splits of every (token, KV head) with more than one split, after all units.  The
// n splits are cut into four consecutive groups of c = ceil(n / 4); every output pair of every
// head is handled by four consecutive lanes, one per group.  Per output, with M = max_s m_s (exact):
//   L_q = sum_{s in group q, ascending} l_s 2^(m_s - M),  A_q = sum_{s in group q} acc_s 2^(m_s - M),
//   L = ((L_0 + L_1) + L_2) + L_3,  A likewise,  o = A / L.
// n depends only on the token's position, so the order is fixed for the token whatever the batch.
// A block covers kMergePairs output pairs of one (token, KV head); a lane loads the (m, l) pairs
// and partial sums of up to kMergeBatch splits of its group in one batch before it uses them, so
// that a context of up to 4 * kMergeBatch splits costs one round of loads.  Two instantiations
// differ only in that batch (and so in registers and blocks per SM): 4 for short split lists,
// where many resident blocks matter, 16 for long ones.  The arithmetic is the same.
constexpr int kMergePairs = kMergeThreads / 4;

template <int D, int G, int kMergeBatch>
__global__ void __launch_bounds__(kMergeThreads, kMergeBatch <= 4 ? 4 : 2) merge_kernel(const Params p) {
  constexpr int kPairs = G * D / 2;
  constexpr int kSlices = (kPairs + kMergePairs - 1) / kMergePairs;
  const int64_t job = blockIdx.x / kSlices;             // token * Hkv + KV head
  const int slice = int(blockIdx.x - job * kSlices);
  const int64_t t = job / p.Hkv;
  const int32_t kh = int32_t(job - t * p.Hkv);
  if (t >= p.T) return;
  // The token's request and position are read before the wait for the attention kernel: that
  // kernel does not write them, and this grid starts only after each of its blocks has passed its
  // own wait for the kernels before it, so they are complete and visible (read from L2).
  const int32_t b = __ldcg(p.q_seq + t), pos = __ldcg(p.q_pos + t);
  if (b < 0 || b >= p.B || pos < 0 || int64_t(pos / p.page_size) >= p.max_pages) return;
  const int32_t n = splits_of(pos, p.split);
  if (n == 1 || pos > p.max_pos) return;    // written directly / refused by the plan
  ptx::grid_dependency_wait();   // every unit's partial results are complete and visible
  const int64_t slot0 = job * int64_t(p.max_splits);
  const int32_t c = (n + 3) / 4;
  const int pr = slice * kMergePairs + int(threadIdx.x >> 2), q = int(threadIdx.x & 3);
  const bool valid = pr < kPairs;                       // uniform over the four lanes of a pair
  const int g = valid ? pr / (D / 2) : 0, d = valid ? (pr % (D / 2)) * 2 : 0;
  const int32_t s0 = min(n, q * c), s1 = valid ? min(n, s0 + c) : s0;
  const float* mlp = p.ml + (slot0 * G + g) * 2;        // split ss: mlp[ss * G * 2]
  const float* pp = p.part + (slot0 * G + g) * D + d;   // split ss: pp[ss * G * D]
  float L = 0.0f, A0 = 0.0f, A1 = 0.0f;
  if (c <= kMergeBatch) {
    float2 ml[kMergeBatch], v[kMergeBatch];
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      if (s0 + i < s1) {
        ml[i] = *reinterpret_cast<const float2*>(mlp + int64_t(s0 + i) * G * 2);
        v[i] = *reinterpret_cast<const float2*>(pp + int64_t(s0 + i) * G * D);
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i)
      if (s0 + i < s1) m = fmaxf(m, ml[i].x);
    const float m1 = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));   // the pair's four lanes
    const float M = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 2));
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      if (s0 + i < s1) {
        const float f = exp2f(__fsub_rn(ml[i].x, M));
        L = __fadd_rn(L, __fmul_rn(ml[i].y, f));
        A0 = __fadd_rn(A0, __fmul_rn(v[i].x, f));
        A1 = __fadd_rn(A1, __fmul_rn(v[i].y, f));
      }
    }
  } else {
    // longer contexts: the group maximum over batches of loads, then the sums batch by batch
    float m = -INFINITY;
    for (int32_t b0 = s0; b0 < s1; b0 += kMergeBatch) {
      float mv[kMergeBatch];
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i)
        mv[i] = b0 + i < s1 ? mlp[int64_t(b0 + i) * G * 2] : -INFINITY;
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i) m = fmaxf(m, mv[i]);
    }
    const float m1 = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));   // the pair's four lanes
    const float M = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 2));
    for (int32_t b0 = s0; b0 < s1; b0 += kMergeBatch) {
      float2 ml[kMergeBatch], v[kMergeBatch];
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i) {
        if (b0 + i < s1) {
          ml[i] = *reinterpret_cast<const float2*>(mlp + int64_t(b0 + i) * G * 2);
          v[i] = *reinterpret_cast<const float2*>(pp + int64_t(b0 + i) * G * D);
        }
      }
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i) {
        if (b0 + i < s1) {
          const float f = exp2f(__fsub_rn(ml[i].x, M));
          L = __fadd_rn(L, __fmul_rn(ml[i].y, f));
          A0 = __fadd_rn(A0, __fmul_rn(v[i].x, f));
          A1 = __fadd_rn(A1, __fmul_rn(v[i].y, f));
        }
      }
    }
  }
  // the four group sums of the pair, added in group order by the pair's first lane
  const int base = int(threadIdx.x & 31) & ~3;
  float Lq[4], A0q[4], A1q[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    Lq[k] = __shfl_sync(0xFFFFFFFFu, L, base + k);
    A0q[k] = __shfl_sync(0xFFFFFFFFu, A0, base + k);
    A1q[k] = __shfl_sync(0xFFFFFFFFu, A1, base + k);
  }
  if (valid && q == 0) {
    const float Ls = __fadd_rn(__fadd_rn(__fadd_rn(Lq[0], Lq[1]), Lq[2]), Lq[3]);
    const float As0 = __fadd_rn(__fadd_rn(__fadd_rn(A0q[0], A0q[1]), A0q[2]), A0q[3]);
    const float As1 = __fadd_rn(__fadd_rn(__fadd_rn(A1q[0], A1q[1]), A1q[2]), A1q[3]);
    *reinterpret_cast<uint32_t*>(p.o + (t * p.Hq + int64_t(kh) * G + g) * D + d) =
        pack_bf16x2(__fdiv_rn(As0, Ls), __fdiv_rn(As1, Ls));
  }
}

template <int D, int G>
constexpr int merge_slices_of() { return (G * D / 2 + kMergePairs - 1) / kMergePairs; }

struct KernelInfo {
  const void* fn = nullptr;
  const void* tma = nullptr;
  const void* fn_inline = nullptr;    // the same kernels deriving unit records themselves
  const void* tma_inline = nullptr;
  const void* tma4 = nullptr;         // the TMA kernels with registers for four blocks per SM
  const void* tma4_inline = nullptr;
  const void* merge = nullptr;        // split lists of up to 4 per group
  const void* merge_long = nullptr;   // longer split lists
  size_t (*smem)(int) = nullptr;
  size_t (*tma_fixed)(int) = nullptr;   // TMA variant: shared memory besides the ring
  int tma_stage_bytes = 0, tma_threads = 0, tma_blocks_per_sm = 0;
  int merge_slices = 1;   // merge blocks per (token, KV head)
};

template <int D, int G>
KernelInfo info() {
  KernelInfo k;
  k.fn = reinterpret_cast<const void*>(&attn_kernel<D, G, false>);
  k.tma = reinterpret_cast<const void*>(&attn_tma_kernel<D, G, false, TmaCfg<D, G>::BLOCKS_PER_SM>);
  k.fn_inline = reinterpret_cast<const void*>(&attn_kernel<D, G, true>);
  k.tma_inline = reinterpret_cast<const void*>(&attn_tma_kernel<D, G, true, TmaCfg<D, G>::BLOCKS_PER_SM>);
  k.tma4 = reinterpret_cast<const void*>(&attn_tma_kernel<D, G, false, 4>);
  k.tma4_inline = reinterpret_cast<const void*>(&attn_tma_kernel<D, G, true, 4>);
  k.tma_fixed = &TmaCfg<D, G>::fixed_bytes;
  k.tma_stage_bytes = TmaCfg<D, G>::STAGE_BYTES;
  k.tma_threads = TmaCfg<D, G>::THREADS;
  k.tma_blocks_per_sm = TmaCfg<D, G>::BLOCKS_PER_SM;
  k.merge = reinterpret_cast<const void*>(&merge_kernel<D, G, 4>);
  k.merge_long = reinterpret_cast<const void*>(&merge_kernel<D, G, 16>);
  k.merge_slices = merge_slices_of<D, G>();
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A cache [rows = num_pages * page_size, Hkv, D] (bf16) as a 3-D tensor, box [page_size, 1, 64]:
// one page's rows of one KV head and 64 of its dimensions, 128-byte swizzled, zero fill outside.
bool encode_cache(CUtensorMap* m, const void* base, int64_t rows, int Hkv, int D, int page_size) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(rows)};
  cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(Hkv) * D * 2};
  cuuint32_t box[3] = {64, 1, cuuint32_t(page_size)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace biattn

struct bi_attention {
  int Hq = 0, Hkv = 0, D = 0, G = 0, page_size = 0, split = 0;
  float scale = 0.0f;
  int device = 0, num_sms = 0, max_ctas = 0;
  size_t smem = 0;
  // TMA page-box variant (page sizes 8, 16, 32, 64): ring depth, shared memory, grid bound
  bool tma = false;
  int nstage = 0, tma_ctas = 0;
  int tma_ctas_inline = 0, max_ctas_inline = 0;   // grid bounds of the kernels deriving their units
  size_t tma_smem = 0;
  // the TMA kernel with registers for four blocks per SM (a shallower ring), for calls that fit
  // in one round of its blocks but not of the three-block kernel's
  bool tma4 = false;
  int nstage4 = 0, tma4_ctas = 0, tma4_ctas_inline = 0;
  size_t tma4_smem = 0;
  biattn::KernelInfo kern;
  uint32_t* d_status = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

namespace {

struct WsLayout {
  size_t cum, urec, part, ml, total;
};

WsLayout layout_of(const bi_attention* h, int64_t T, int64_t max_pos) {
  const int64_t max_splits = max_pos / h->split + 1;
  const int64_t slots = T * h->Hkv * max_splits;
  WsLayout w;
  w.cum = 0;
  w.urec = biattn::align256(size_t(T + 1) * sizeof(int32_t));
  w.part = w.urec + biattn::align256(size_t(slots) * sizeof(int4));
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
  const size_t smem = k.smem(int(split));
  // The attribute is per kernel, shared by every handle of the same head shape: set the largest
  // any handle of this kernel can need (split 1024).
  const size_t smem_cap = k.smem(1024);
  if (smem_cap > 232448) return BI_GEMM_ERR_UNSUPPORTED;
  int per_sm_inline = 0;
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_cap)) != cudaSuccess ||
      cudaFuncSetAttribute(k.fn_inline, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_cap)) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, biattn::kThreads, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_inline, k.fn_inline, biattn::kThreads, smem) !=
          cudaSuccess ||
      per_sm < 1 || per_sm_inline < 1) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  // TMA variant: the deepest ring (up to 8 stages) with which its blocks per SM fit
  bool tma = false;
  int nstage = 0, tma_per_sm = 0, tma_per_sm_inline = 0;
  int nstage4 = 0, tma4_per_sm = 0, tma4_per_sm_inline = 0;
  size_t tma_smem = 0, tma4_smem = 0;
  if (page_size == 8 || page_size == 16 || page_size == 32 || page_size == 64) {
    int sm_bytes = 0, reserved = 0, optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, k.tma) != cudaSuccess) {
      cudaGetLastError();
      return BI_GEMM_ERR_CUDA;
    }
    const int64_t budget = int64_t(sm_bytes) / k.tma_blocks_per_sm - reserved - int64_t(fa.sharedSizeBytes) -
                           int64_t(k.tma_fixed(int(split)));
    nstage = int(std::min<int64_t>(biattn::kTmaMaxStages, budget / (k.tma_stage_bytes + 16)));
    if (nstage >= 2 && biattn::encode_fn()) {
      tma_smem = k.tma_fixed(int(split)) + size_t(nstage) * (k.tma_stage_bytes + 16);
      // per kernel, shared by every handle of the head shape: the most a block may have
      if (cudaFuncSetAttribute(k.tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               optin - int(fa.sharedSizeBytes)) != cudaSuccess ||
          cudaFuncSetAttribute(k.tma_inline, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               optin - int(fa.sharedSizeBytes)) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&tma_per_sm, k.tma, k.tma_threads, tma_smem) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&tma_per_sm_inline, k.tma_inline, k.tma_threads,
                                                        tma_smem) != cudaSuccess) {
        cudaGetLastError();
        return BI_GEMM_ERR_CUDA;
      }
      tma = tma_per_sm >= 1 && tma_per_sm_inline >= 1;
    }
    // the same kernel with registers for four blocks per SM and the ring that four leave room for
    cudaFuncAttributes fa4;
    if (tma && cudaFuncGetAttributes(&fa4, k.tma4) == cudaSuccess) {
      const int64_t budget4 = int64_t(sm_bytes) / 4 - reserved - int64_t(fa4.sharedSizeBytes) -
                              int64_t(k.tma_fixed(int(split)));
      nstage4 = int(std::min<int64_t>(biattn::kTmaMaxStages, budget4 / (k.tma_stage_bytes + 16)));
      if (nstage4 >= 2) {
        tma4_smem = k.tma_fixed(int(split)) + size_t(nstage4) * (k.tma_stage_bytes + 16);
        if (cudaFuncSetAttribute(k.tma4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - int(fa4.sharedSizeBytes)) != cudaSuccess ||
            cudaFuncSetAttribute(k.tma4_inline, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin - int(fa4.sharedSizeBytes)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&tma4_per_sm, k.tma4, k.tma_threads, tma4_smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&tma4_per_sm_inline, k.tma4_inline, k.tma_threads,
                                                          tma4_smem) != cudaSuccess) {
          cudaGetLastError();
          return BI_GEMM_ERR_CUDA;
        }
      }
    }
    cudaGetLastError();
  }
  bi_attention* h = new (std::nothrow) bi_attention();
  if (!h) return BI_GEMM_ERR_OOM;
  h->tma = tma;
  h->nstage = tma ? nstage : 0;
  h->tma_smem = tma_smem;
  h->tma_ctas = tma_per_sm * sms;
  h->tma_ctas_inline = tma_per_sm_inline * sms;
  h->max_ctas_inline = per_sm_inline * sms;
  // the four-block kernel only where it fits more blocks per SM than the three-block one
  h->tma4 = tma && nstage4 >= 2 && tma4_per_sm > tma_per_sm && tma4_per_sm_inline > tma_per_sm_inline;
  h->nstage4 = h->tma4 ? nstage4 : 0;
  h->tma4_smem = tma4_smem;
  h->tma4_ctas = h->tma4 ? tma4_per_sm * sms : 0;
  h->tma4_ctas_inline = h->tma4 ? tma4_per_sm_inline * sms : 0;
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

namespace {

// bi_attention_run with the failure injection of the test controls (stall_block >= 0: that
// block of the TMA kernel never issues its first load), the limit of the ring waits, and the
// kernel choice (0: automatic; 1: the TMA page-box kernel where the handle has it; 2: the
// row-copy kernel), which the test controls use to run both kernels on the same calls.
int attention_run(bi_attention* h, const void* q, int64_t T, const int32_t* q_seq, const int32_t* q_pos,
                  const void* k_cache, const void* v_cache, int64_t num_pages, const int32_t* page_table,
                  int64_t num_seqs, int64_t max_pages, int64_t max_pos, void* o, void* stream, int32_t stall_block,
                  uint64_t timeout_ns, int32_t kernel_choice = 0) {
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
  p.urec = reinterpret_cast<int4*>(ws + w.urec);
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
  p.max_pos = int32_t(max_pos);
  p.c = h->scale * 1.4426950408889634f;   // log2(e)
  p.nstage = h->nstage;
  p.stall_block = stall_block;
  p.timeout_ns = timeout_ns;
  // The TMA variant needs the caches' rows addressable by int32 box coordinates (one page past
  // the end included); otherwise, or if a tensor map cannot be encoded, the row-copy kernel
  // runs: both give the same bits.
  CUtensorMap tmk, tmv;
  const int64_t rows = num_pages * h->page_size;
  // Small batches derive the unit records inside the attention kernel (same numbering), which
  // saves the plan launch and its wait; larger ones read the plan's table.
  p.inline_plan = T <= biattn::kInlinePlanMaxT ? 1 : 0;
  // A call whose units fit in one round of the row-copy kernel's (more numerous, smaller) blocks
  // but not in one round of either TMA kernel's runs the row-copy kernel: the second round of a
  // few units would otherwise run alone at one block per SM.  A call that fits in one round of
  // the four-block TMA kernel but not of the three-block one runs the four-block kernel (its
  // shallower ring costs less than a second round).  All give the same bits.
  const int64_t units_all = T * h->Hkv * int64_t(p.max_splits);
  const bool inl = p.inline_plan != 0;
  const int64_t tma3_slots = inl ? h->tma_ctas_inline : h->tma_ctas;
  const int64_t tma4_slots = h->tma4 ? (inl ? h->tma4_ctas_inline : h->tma4_ctas) : 0;
  const bool one_round_rows = units_all > std::max(tma3_slots, tma4_slots) &&
                              units_all <= (inl ? h->max_ctas_inline : h->max_ctas);
  const bool want_tma = kernel_choice == 1 || (kernel_choice == 0 && !one_round_rows);
  const bool use_tma = h->tma && want_tma && num_pages > 0 && rows + h->page_size < (int64_t(1) << 31) &&
                       biattn::encode_cache(&tmk, k_cache, rows, h->Hkv, h->D, h->page_size) &&
                       biattn::encode_cache(&tmv, v_cache, rows, h->Hkv, h->D, h->page_size);
  if (!p.inline_plan) {
    biattn::plan_kernel<<<1, 1024, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return BI_GEMM_ERR_CUDA;
  }
  const int64_t units = T * h->Hkv * int64_t(p.max_splits);
  void* args[1] = {&p};
  void* targs[3] = {&tmk, &tmv, &p};
  // the attention and merge kernels are launched as programmatic dependents: each may start
  // while its predecessor runs and waits (griddepcontrol.wait) before it reads what that wrote
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool use_tma4 = use_tma && units_all > tma3_slots && units_all <= tma4_slots;
  if (use_tma) {
    cfg.gridDim = dim3(unsigned(std::min<int64_t>(units, use_tma4 ? tma4_slots : tma3_slots)));
    cfg.blockDim = dim3(h->kern.tma_threads);
    cfg.dynamicSmemBytes = use_tma4 ? h->tma4_smem : h->tma_smem;
    p.nstage = use_tma4 ? h->nstage4 : h->nstage;
  } else {
    cfg.gridDim = dim3(unsigned(std::min<int64_t>(units, inl ? h->max_ctas_inline : h->max_ctas)));
    cfg.blockDim = dim3(biattn::kThreads);
    cfg.dynamicSmemBytes = h->smem;
  }
  const void* fn = use_tma ? (use_tma4 ? (inl ? h->kern.tma4_inline : h->kern.tma4)
                                       : (inl ? h->kern.tma_inline : h->kern.tma))
                           : (inl ? h->kern.fn_inline : h->kern.fn);
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, use_tma ? targs : args);
  if (e == cudaSuccess) {
    cfg.gridDim = dim3(unsigned(T * h->Hkv * h->kern.merge_slices));
    cfg.blockDim = dim3(biattn::kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    // at most four splits per group: the instantiation with more resident blocks
    e = cudaLaunchKernelExC(&cfg, (p.max_splits + 3) / 4 <= 4 ? h->kern.merge : h->kern.merge_long, args);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  return BI_GEMM_OK;
}

}  // namespace

BI_GEMM_API int bi_attention_run(bi_attention_t h, const void* q, int64_t T, const int32_t* q_seq,
                                 const int32_t* q_pos, const void* k_cache, const void* v_cache,
                                 int64_t num_pages, const int32_t* page_table, int64_t num_seqs,
                                 int64_t max_pages, int64_t max_pos, void* o, void* stream) {
  return attention_run(h, q, T, q_seq, q_pos, k_cache, v_cache, num_pages, page_table, num_seqs, max_pages, max_pos,
                       o, stream, -1, biattn::kTimeoutNs);
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
  return (s & biattn::kErrTimeout) ? BI_GEMM_ERR_TIMEOUT : BI_GEMM_ERR_INVALID_ARG;
}

BI_GEMM_API int bi_attention_get_config(bi_attention_t h, bi_attention_config* c) {
  if (!h || !c) return BI_GEMM_ERR_INVALID_ARG;
  c->num_q_heads = h->Hq;
  c->num_kv_heads = h->Hkv;
  c->head_dim = h->D;
  c->page_size = h->page_size;
  c->split_size = h->split;
  c->threads = h->tma ? h->kern.tma_threads : biattn::kThreads;
  c->stage_positions = biattn::kStagePos;
  c->max_ctas = h->tma ? h->tma_ctas : h->max_ctas;
  c->num_sms = h->num_sms;
  c->tma_pages = h->tma ? 1 : 0;
  c->ring_stages = h->tma ? h->nstage : biattn::kStages;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_attention_destroy(bi_attention_t h) {
  if (!h) return BI_GEMM_OK;
  if (h->ws) cudaFree(h->ws);
  if (h->d_status) cudaFree(h->d_status);
  delete h;
  return BI_GEMM_OK;
}
