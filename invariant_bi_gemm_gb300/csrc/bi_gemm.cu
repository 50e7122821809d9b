// bi_gemm.cu — host side of the batch-invariant GEMM: configuration at create, tensor maps,
// workspace, launch, status word.  Implements include/bi_gemm.h.
//
// The configuration rule ("Batch-invariant matrix multiplication", nondeterminism article:
// compile one kernel configuration and use it for all shapes; strategy switches keyed on
// the block/SM ratio are where libraries lose invariance):
//   tile      128 x BN, BN = 64 / 128 / 256 (bf16) or 128 / 256 (MXFP8) from N alone; with
//             BN = 256 the tile is 256 x 256 on a CTA pair (cta_group::2);
//   MMA       tcgen05.mma M=128 (M=256 on a pair), N=BN, K=16 (bf16) or K=32 (MXFP8);
//   K stage   128 bytes of K per stage (64 bf16 / 128 E4M3), ascending k-blocks;
//   split S   1, except for a single N tile (N <= BN) with a long K, where
//             S = min(32, pow2floor(SMs / 4), pow2floor(KB / 8)) — the pinned
//             "min(cap, n_sms // 4) rounded down to a power of two" of "[BI][DSv4] Make mHC
//             tilelang ops batch invariant" ("What"), with each split keeping >= 8 k-blocks.
// None of these reads M.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>

#include "../../include/bi_gemm.h"
#include "bi_gemm_kernel.cuh"

#ifndef BI_GEMM_API
#define BI_GEMM_API extern "C" __attribute__((visibility("default")))
#endif

namespace bigemm {

constexpr int kVersion = (1 << 16) | 0;
constexpr int64_t kCoopMergeBytes = 24 << 10;   // partial bytes of a sub-tile above which its
                                                // split CTAs share the merge
constexpr uint64_t kDefaultTimeoutNs = 5ull * 1000 * 1000 * 1000;
// Raster order (visiting order only; it decides no arithmetic): while x fits comfortably in L2
// the M tiles vary fastest (x stays resident, W streams once); a larger x is visited in groups
// of 16 N tiles, so that the W slabs of a group (16 x K x 256 x 2 bytes) stay resident while x
// is re-read once per group.
constexpr int64_t kRasterXResidentBytes = int64_t(40) << 20;
constexpr int64_t kRasterGroupN = 16;

// ------------------------------------------------------------------ kernel table

struct KernelInfo {
  const void* fn = nullptr;
  int threads = 0, smem = 0, tmem_cols = 0, stages = 0, bn = 0, bk = 0, mma_k = 0, ctas = 1;
  int w_box_cols = 0, w_swizzle = 128;   // TMA box width of W (columns) and its swizzle span
  bool smallm = false;                   // has the small-M pipeline (bf16 pair tile)
  int ring_bytes = 0, b_bytes = 0;       // its ring and one W tile (bytes per CTA)
};

template <class C>
KernelInfo info_of() {
  KernelInfo k;
  k.fn = reinterpret_cast<const void*>(&bi_gemm_kernel<C>);
  k.threads = C::THREADS;
  k.smem = C::SMEM_BYTES;
  k.tmem_cols = C::TMEM_COLS;
  k.stages = C::STAGES;
  k.bn = C::BN;
  k.bk = C::BK;
  k.mma_k = C::MMA_K;
  k.ctas = C::CTAS;
  k.w_box_cols = C::ATOM_N;
  k.w_swizzle = C::B_SW;
  k.smallm = C::SMALLM;
  k.ring_bytes = C::RING_BYTES;
  k.b_bytes = C::B_BYTES;
  return k;
}

// Pipeline depth of the CTA-pair tile (a stage: 16 KB of x and 16 KB of W per CTA).
#ifndef BI_GEMM_PAIR_STAGES
#define BI_GEMM_PAIR_STAGES 6
#endif
// Pipeline depth of the MXFP8 pair tile (a stage: 16 KB of x, 16 KB of W and 1.5 KB of scales
// per CTA; one accumulator, since 256 fp32 columns plus the scale columns fill the TMEM).
#ifndef BI_GEMM_FP8_PAIR_STAGES
#define BI_GEMM_FP8_PAIR_STAGES 6
#endif

// dtype 0/1: bf16 in, bf16/f32 out; dtype 2: MXFP8 in, bf16 out.
static KernelInfo select_kernel(int dtype, int bn) {
  switch (dtype) {
    case BI_BF16_OUT_BF16:
      if (bn == 64) return info_of<KCfg<false, false, 64, 8, 2>>();
      if (bn == 128) return info_of<KCfg<false, false, 128, 6, 2>>();
      return info_of<KCfg<false, false, 256, BI_GEMM_PAIR_STAGES, 2, 2>>();
    case BI_BF16_OUT_F32:
      if (bn == 64) return info_of<KCfg<false, true, 64, 8, 2>>();
      if (bn == 128) return info_of<KCfg<false, true, 128, 6, 2>>();
      return info_of<KCfg<false, true, 256, BI_GEMM_PAIR_STAGES, 2, 2>>();
    default:
      if (bn == 128) return info_of<KCfg<true, false, 128, 6, 2>>();
      return info_of<KCfg<true, false, 256, BI_GEMM_FP8_PAIR_STAGES, 1, 2>>();
  }
}

static int pow2_floor(int64_t v) {
  int p = 1;
  while ((int64_t)p * 2 <= v) p *= 2;
  return v >= 1 ? p : 0;
}

// ------------------------------------------------------------------ tensor-map encoder

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major [rows, cols] tensor of 1-, 2- or 4-byte elements (uint8 / bf16 / fp32), box
// [box_rows, box_cols], 128- or 64-byte swizzle (0 = none), zero fill for loads.
static bool encode_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, uint32_t box_cols, int swizzle = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t elem = uint64_t(elem_bytes);
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUtensorMapSwizzle sw = swizzle == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace bigemm

using namespace bigemm;

struct bi_gemm {
  int64_t K = 0, N = 0;
  int dtype = 0, scale_layout = 0;
  int device = 0, num_sms = 0, max_ctas = 0;
  int split = 1, kblocks = 0, n_tiles = 0;
  int max_groups = 0;      // CTA groups (single CTAs or pairs) resident at once
  uint32_t flags = 0;      // BI_GEMM_FLAG_*
  uint64_t timeout_ns = kDefaultTimeoutNs;
  KernelInfo kern;
  uint32_t* d_status = nullptr;
  // split-K workspace: [arrival counters, cap_tiles x 4 B, padded to 256 B][fp32 partials]
  void* ws = nullptr;
  int64_t ws_cap_tiles = 0;
  size_t ws_cap_part = 0;
  bool ws_dirty = false;
  // W tensor map cache
  const void* w_cached = nullptr;
  CUtensorMap tmap_w;
  std::mutex mu;
};

namespace {

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int64_t K, int64_t N, int dtype, int scale_layout) {
  if (dtype < BI_BF16_OUT_BF16 || dtype > BI_MXFP8E4M3_OUT_BF16) return BI_GEMM_ERR_INVALID_ARG;
  if (scale_layout != BI_SCALES_NONE && scale_layout != BI_SCALES_E8M0_K32)
    return BI_GEMM_ERR_INVALID_ARG;
  if (K < 0 || N < 0) return BI_GEMM_ERR_INVALID_ARG;
  if (K == 0 || N == 0 || K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31))
    return BI_GEMM_ERR_UNSUPPORTED;
  if (dtype == BI_MXFP8E4M3_OUT_BF16) {
    if (scale_layout != BI_SCALES_E8M0_K32) return BI_GEMM_ERR_UNSUPPORTED;
    if (K % 128 != 0 || N % 16 != 0) return BI_GEMM_ERR_UNSUPPORTED;
  } else {
    if (scale_layout != BI_SCALES_NONE) return BI_GEMM_ERR_UNSUPPORTED;
    if (K % 8 != 0 || N % 8 != 0) return BI_GEMM_ERR_UNSUPPORTED;
  }
  return BI_GEMM_OK;
}

// Tile width from N alone: 64 / 128 for narrow N, else 256 (on a CTA pair for bf16).  (A
// 192-wide pair tile, which would fill all 76 pairs at N = 14336, was measured slower at every
// M on GB300: its 96-column W halves need 64-byte swizzle rows.)
int block_n_for(int64_t N, int dtype, int /*num_sms*/) {
  if (dtype == BI_MXFP8E4M3_OUT_BF16) return N <= 128 ? 128 : 256;
  return N <= 64 ? 64 : (N <= 128 ? 128 : 256);
}

int auto_split(int64_t n_tiles, int64_t kblocks, int num_sms) {
  if (n_tiles != 1) return 1;
  int s = std::min(32, std::min(pow2_floor(num_sms / 4), pow2_floor(kblocks / 8)));
  return std::max(1, s);
}

size_t counters_bytes(int64_t tiles) { return (size_t(tiles) * sizeof(uint32_t) + 255) & ~size_t(255); }

// Make the workspace hold `tiles` counters (all zero) and tiles*split partial tiles.
int ensure_workspace(bi_gemm* h, int64_t tiles, int split, cudaStream_t st) {
  if (split <= 1) return BI_GEMM_OK;
  const size_t part = size_t(tiles) * split * kBM * h->kern.bn * sizeof(float);
  if (h->ws && tiles <= h->ws_cap_tiles && part <= h->ws_cap_part) {
    if (h->ws_dirty) {
      if (cudaMemsetAsync(h->ws, 0, counters_bytes(h->ws_cap_tiles), st) != cudaSuccess)
        return BI_GEMM_ERR_CUDA;
      h->ws_dirty = false;
    }
    return BI_GEMM_OK;
  }
  const int64_t cap_tiles = std::max(tiles, h->ws_cap_tiles);
  const size_t cap_part = std::max(part, h->ws_cap_part);
  if (h->ws) {
    cudaFreeAsync(h->ws, st);
    h->ws = nullptr;
    h->ws_cap_tiles = 0;
    h->ws_cap_part = 0;
  }
  void* p = nullptr;
  if (cudaMallocAsync(&p, counters_bytes(cap_tiles) + cap_part, st) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_OOM;
  }
  if (cudaMemsetAsync(p, 0, counters_bytes(cap_tiles), st) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeAsync(p, st);
    return BI_GEMM_ERR_CUDA;
  }
  h->ws = p;
  h->ws_cap_tiles = cap_tiles;
  h->ws_cap_part = cap_part;
  h->ws_dirty = false;
  return BI_GEMM_OK;
}

struct Shape {
  int64_t m_tiles, tiles, subtiles;   // output tiles of TILE_M rows; 128-row sub-tiles
};

Shape shape_of(const bi_gemm* h, int64_t M) {
  Shape sh;
  const int64_t tile_m = int64_t(kBM) * h->kern.ctas;
  sh.m_tiles = (M + tile_m - 1) / tile_m;
  sh.tiles = sh.m_tiles * h->n_tiles;
  sh.subtiles = sh.tiles * h->kern.ctas;
  return sh;
}

// Encode the tensor maps, fill the kernel parameters and launch.  `ws` / `counters` are the
// split-K scratch (ignored when split == 1).
int launch_core(bi_gemm* h, const void* x, int64_t M, const void* W, const bi_gemm_scales* scales,
                void* y, cudaStream_t st, int split, float* ws, uint32_t* counters,
                uint32_t test_flags) {
  const bool fp8 = h->dtype == BI_MXFP8E4M3_OUT_BF16;
  const Shape sh = shape_of(h, M);
  if (sh.tiles * split >= (int64_t(1) << 31)) return BI_GEMM_ERR_UNSUPPORTED;

  // x box: 128 rows, or only round_up(M, 8) rows when M < 128 (rows past M are never stored)
  const uint32_t a_box_rows = M >= kBM ? uint32_t(kBM) : uint32_t((M + 7) / 8 * 8);
  CUtensorMap tmap_x, tmap_y;
  if (!encode_2d(&tmap_x, x, fp8 ? 1 : 2, uint64_t(M), uint64_t(h->K), a_box_rows, 128 / (fp8 ? 1 : 2)))
    return BI_GEMM_ERR_CUDA;
  // y: 32 x 32 output blocks staged with the swizzle that matches their row length
  // (bf16: 64-byte rows, 64-byte swizzle; fp32: 128-byte rows, 128-byte swizzle)
  const bool f32 = h->dtype == BI_BF16_OUT_F32;
  if (!encode_2d(&tmap_y, y, f32 ? 4 : 2, uint64_t(M), uint64_t(h->N), 32, 32, f32 ? 128 : 64))
    return BI_GEMM_ERR_CUDA;
  if (h->w_cached != W) {
    if (!encode_2d(&h->tmap_w, W, fp8 ? 1 : 2, uint64_t(h->K), uint64_t(h->N), h->kern.bk,
                   uint32_t(h->kern.w_box_cols), h->kern.w_swizzle)) {
      h->w_cached = nullptr;
      return BI_GEMM_ERR_CUDA;
    }
    h->w_cached = W;
  }

  KParams p;
  std::memset(&p, 0, sizeof(p));
  p.y = y;
  p.sx = scales ? scales->sx : nullptr;
  p.sw = scales ? scales->sw : nullptr;
  p.ws = split > 1 ? ws : nullptr;
  p.counters = split > 1 ? counters : nullptr;
  p.status = h->d_status;
  p.M = int32_t(M);
  p.N = int32_t(h->N);
  p.K = int32_t(h->K);
  p.m_tiles = int32_t(sh.m_tiles);
  p.n_tiles = int32_t(h->n_tiles);
  p.splits = split;
  p.kblocks = h->kblocks;
  p.a_box_rows = int32_t(a_box_rows);
  const int64_t x_bytes = M * h->K * (fp8 ? 1 : 2);
  p.group_n = int32_t(x_bytes <= kRasterXResidentBytes ? 1 : std::min<int64_t>(kRasterGroupN, h->n_tiles));
  p.w_early = (h->flags & BI_GEMM_FLAG_STATIC_W) ? 1 : 0;
  // Small M on the pair tile (an x box of at most 64 rows): stages of two k-blocks laid out from
  // the x box's rows, as many as the ring holds (at most STAGES - 1), keeping an MMA's 128-row x
  // read of the last slot inside the ring.  A pipeline choice: no instruction, operand or order
  // changes.
  if (h->kern.smallm && a_box_rows <= 64) {
    const int slot = int(a_box_rows) * 128 + h->kern.b_bytes;
    int st = std::min(h->kern.stages - 1, h->kern.ring_bytes / (2 * slot));
    while (st > 2 && (2 * st - 1) * slot + kBM * 128 > h->kern.ring_bytes) --st;
    if (st >= 2 && (2 * st - 1) * slot + kBM * 128 <= h->kern.ring_bytes) {
      p.small_m = 1;
      p.small_stages = st;
      p.slot_bytes = uint32_t(slot);
    }
  }
  p.timeout_ns = h->timeout_ns;
  p.test_flags = test_flags;

  const int64_t units = sh.tiles * split;
  const int groups = int(std::min<int64_t>(units, h->max_groups));
  // The split CTAs of a 128-row sub-tile share its merge when every unit has its own resident
  // CTA group (so they can wait for each other) and the partials of the sub-tile are more than
  // one CTA reads faster than the S CTAs can meet (kCoopMergeBytes, measured on GB300);
  // otherwise the last CTA to arrive merges alone.  Either way every element is summed in split
  // order, so this choice moves data, not arithmetic.
  const int64_t merge_items = std::min<int64_t>(M, kBM) * ((std::min<int64_t>(h->N, h->kern.bn) + 3) / 4);
  p.coop_merge =
      (split > 1 && units <= h->max_groups && merge_items * split * 16 > kCoopMergeBytes) ? 1 : 0;
  void* args[4] = {&tmap_x, &h->tmap_w, &tmap_y, &p};
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(unsigned(groups * h->kern.ctas));
  cfg.blockDim = dim3(unsigned(h->kern.threads));
  cfg.dynamicSmemBytes = size_t(h->kern.smem);
  cfg.stream = st;
  // Programmatic dependent launch: the kernel's set-up may overlap the previous kernel's tail;
  // it waits (griddepcontrol.wait) for that kernel to complete before touching global memory.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (h->kern.ctas > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(h->kern.ctas);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  if (cudaLaunchKernelExC(&cfg, h->kern.fn, args) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  return BI_GEMM_OK;
}

// Launch one run with the handle's workspace; `split_override` > 0 replaces the handle's split
// count (control build only).
int launch(bi_gemm* h, const void* x, int64_t M, const void* W, const bi_gemm_scales* scales,
           void* y, cudaStream_t st, int split_override, uint32_t test_flags) {
  const int split = split_override > 0 ? split_override : h->split;
  const Shape sh = shape_of(h, M);
  int rc = ensure_workspace(h, sh.subtiles, split, st);
  if (rc != BI_GEMM_OK) return rc;
  uint32_t* counters = split > 1 ? static_cast<uint32_t*>(h->ws) : nullptr;
  float* ws = split > 1 ? reinterpret_cast<float*>(static_cast<char*>(h->ws) + counters_bytes(h->ws_cap_tiles))
                        : nullptr;
  return launch_core(h, x, M, W, scales, y, st, split, ws, counters, test_flags);
}

int validate_run(bi_gemm* h, const void* x, int64_t M, const void* W, const bi_gemm_scales* scales,
                 void* y) {
  if (!h || M < 0) return BI_GEMM_ERR_INVALID_ARG;
  if (M == 0) return BI_GEMM_OK;
  if (M >= (int64_t(1) << 31)) return BI_GEMM_ERR_UNSUPPORTED;
  if (!x || !W || !y) return BI_GEMM_ERR_INVALID_ARG;
  if (!is_aligned(x, 16) || !is_aligned(W, 16) || !is_aligned(y, 16)) return BI_GEMM_ERR_ALIGNMENT;
  if (h->dtype == BI_MXFP8E4M3_OUT_BF16) {
    if (!scales || !scales->sx || !scales->sw) return BI_GEMM_ERR_INVALID_ARG;
    if (!is_aligned(scales->sx, 4) || !is_aligned(scales->sw, 16)) return BI_GEMM_ERR_ALIGNMENT;
  } else if (scales && (scales->sx || scales->sw)) {
    return BI_GEMM_ERR_INVALID_ARG;
  }
  return BI_GEMM_OK;
}

}  // namespace

BI_GEMM_API int bi_gemm_create_ex(bi_gemm_t* out, int64_t K, int64_t N, int dtype,
                                  int scale_layout, const bi_gemm_options* opt) {
  if (!out) return BI_GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = check_shape(K, N, dtype, scale_layout);
  if (rc != BI_GEMM_OK) return rc;
  const int bk = dtype == BI_MXFP8E4M3_OUT_BF16 ? 128 : 64;
  const int64_t kblocks = (K + bk - 1) / bk;
  if (opt && (opt->split_k < 0 || opt->split_k > kblocks || opt->max_ctas < 0 ||
              (opt->flags & ~BI_GEMM_FLAG_STATIC_W) != 0u || opt->reserved != 0u))
    return BI_GEMM_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return BI_GEMM_ERR_UNSUPPORTED;
  if (!encode_fn()) return BI_GEMM_ERR_CUDA;
  const int bn = block_n_for(N, dtype, sms);
  const int64_t n_tiles = (N + bn - 1) / bn;

  bi_gemm* h = new (std::nothrow) bi_gemm();
  if (!h) return BI_GEMM_ERR_OOM;
  h->K = K;
  h->N = N;
  h->dtype = dtype;
  h->scale_layout = scale_layout;
  h->device = dev;
  h->num_sms = sms;
  h->kern = select_kernel(dtype, bn);
  h->max_ctas = (opt && opt->max_ctas > 0) ? std::min(opt->max_ctas, sms) : sms;
  h->max_ctas = std::max(h->max_ctas, h->kern.ctas);
  h->kblocks = int(kblocks);
  h->n_tiles = int(n_tiles);
  h->split = (opt && opt->split_k > 0) ? opt->split_k : auto_split(n_tiles, kblocks, sms);
  h->timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
  h->flags = opt ? opt->flags : 0u;
  if (cudaFuncSetAttribute(h->kern.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, h->kern.smem) !=
          cudaSuccess ||
      cudaMalloc(&h->d_status, sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(h->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    if (h->d_status) cudaFree(h->d_status);
    delete h;
    return BI_GEMM_ERR_CUDA;
  }
  h->max_groups = h->max_ctas / h->kern.ctas;
  if (h->kern.ctas > 1) {
    // pairs that can be resident at once (one pair per two SMs unless the GPCs say otherwise)
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(unsigned(sms));
    cfg.blockDim = dim3(unsigned(h->kern.threads));
    cfg.dynamicSmemBytes = size_t(h->kern.smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(h->kern.ctas);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, h->kern.fn, &cfg) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      cudaFree(h->d_status);
      delete h;
      return BI_GEMM_ERR_UNSUPPORTED;
    }
    h->max_groups = std::max(1, std::min(h->max_groups, clusters));
  }
  *out = h;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_gemm_create(bi_gemm_t* out, int64_t K, int64_t N, int dtype, int scale_layout) {
  return bi_gemm_create_ex(out, K, N, dtype, scale_layout, nullptr);
}

BI_GEMM_API int bi_gemm_run(bi_gemm_t h, const void* x, int64_t M, const void* W,
                            const bi_gemm_scales* scales, void* y, void* stream) {
  int rc = validate_run(h, x, M, W, scales, y);
  if (rc != BI_GEMM_OK || M == 0) return rc;
  std::lock_guard<std::mutex> lk(h->mu);
  return launch(h, x, M, W, scales, y, static_cast<cudaStream_t>(stream), 0, 0u);
}

BI_GEMM_API int bi_gemm_get_device_error(bi_gemm_t h, void* stream) {
  if (!h) return BI_GEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(h->mu);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemcpy(&v, h->d_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (v != 0) {
    if (cudaMemset(h->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
      cudaGetLastError();
      return BI_GEMM_ERR_CUDA;
    }
    h->ws_dirty = true;   // an aborted split run may leave arrival counters non-zero
    return BI_GEMM_ERR_TIMEOUT;
  }
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_gemm_destroy(bi_gemm_t h) {
  if (!h) return BI_GEMM_OK;
  cudaDeviceSynchronize();
  if (h->ws) cudaFree(h->ws);
  if (h->d_status) cudaFree(h->d_status);
  cudaGetLastError();
  delete h;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_gemm_get_config(bi_gemm_t h, bi_gemm_config* c) {
  if (!h || !c) return BI_GEMM_ERR_INVALID_ARG;
  c->block_m = kBM * h->kern.ctas;
  c->block_n = h->kern.bn;
  c->block_k = h->kern.bk;
  c->mma_m = kBM * h->kern.ctas;
  c->mma_n = h->kern.bn;
  c->mma_k = h->kern.mma_k;
  c->stages = h->kern.stages;
  c->split_k = h->split;
  c->num_sms = h->num_sms;
  c->max_ctas = h->max_ctas;
  c->threads = h->kern.threads;
  c->smem_bytes = h->kern.smem;
  c->tmem_cols = h->kern.tmem_cols;
  c->ctas_per_tile = h->kern.ctas;
  c->max_groups = h->max_groups;
  return BI_GEMM_OK;
}

BI_GEMM_API int bi_gemm_workspace_size(bi_gemm_t h, int64_t M, uint64_t* bytes) {
  if (!h || !bytes || M < 0) return BI_GEMM_ERR_INVALID_ARG;
  if (h->split <= 1 || M == 0) {
    *bytes = 0;
    return BI_GEMM_OK;
  }
  const int64_t tiles = shape_of(h, M).subtiles;
  *bytes = counters_bytes(tiles) + size_t(tiles) * h->split * kBM * h->kern.bn * sizeof(float);
  return BI_GEMM_OK;
}

// ------------------------------------------------------------------ gather + GEMM

namespace bigemm {

constexpr int kGatherMaxBlocks = 256;
constexpr int kGatherThreads = 256;

struct GatherParams {
  const void* src[kGatherMaxBlocks];
  int64_t off[kGatherMaxBlocks + 1];   // byte offset of each block in the destination
  void* dst;
};

// Copy every block's bytes to its offset in dst: grid.y is the block, grid.x strides over its
// bytes in 16-byte words (kWord = 16) or 4-byte words (kWord = 4; the MXFP8 scales, whose rows
// are K/32 bytes).  A pure copy: HBM-bound, coalesced, no arithmetic.
template <int kWord>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const __grid_constant__ GatherParams g) {
  using W = typename std::conditional<kWord == 16, uint4, uint32_t>::type;
  const int b = int(blockIdx.y);
  const int64_t n = (g.off[b + 1] - g.off[b]) / kWord;
  const W* src = static_cast<const W*>(g.src[b]);
  W* dst = reinterpret_cast<W*>(static_cast<char*>(g.dst) + g.off[b]);
  ptx::grid_dependency_wait();   // the blocks may be the previous kernel's output
  for (int64_t i = int64_t(blockIdx.x) * kGatherThreads + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * kGatherThreads)
    dst[i] = src[i];
}

}  // namespace bigemm

namespace {

int launch_gather(const void* const* srcs, const int64_t* bytes, int nb, void* dst, int word, int sms,
                  cudaStream_t st) {
  GatherParams g;
  std::memset(&g, 0, sizeof(g));
  int64_t mx = 0;
  g.off[0] = 0;
  for (int b = 0; b < nb; ++b) {
    g.src[b] = srcs[b];
    g.off[b + 1] = g.off[b] + bytes[b];
    mx = std::max(mx, bytes[b]);
  }
  g.dst = dst;
  if (mx == 0) return BI_GEMM_OK;
  const int64_t words = mx / word;
  const int64_t per_block = std::max<int64_t>(1, (int64_t(2) * sms + nb - 1) / nb);   // ~2 CTAs per SM
  const unsigned gx = unsigned(std::min<int64_t>(per_block, (words + kGatherThreads - 1) / kGatherThreads));
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(std::max(1u, gx), unsigned(nb));
  cfg.blockDim = dim3(kGatherThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[1] = {&g};
  const void* fn = word == 16 ? reinterpret_cast<const void*>(&gather_kernel<16>)
                              : reinterpret_cast<const void*>(&gather_kernel<4>);
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  return BI_GEMM_OK;
}

}  // namespace

BI_GEMM_API int bi_gemm_run_gathered(bi_gemm_t h, const bi_gemm_block* blocks, int32_t nblocks, void* x_out,
                                     uint8_t* sx_out, const void* W, const uint8_t* sw, void* y, void* stream) {
  if (!h || !blocks || nblocks < 1 || nblocks > kGatherMaxBlocks) return BI_GEMM_ERR_INVALID_ARG;
  const bool fp8 = h->dtype == BI_MXFP8E4M3_OUT_BF16;
  const int64_t xrow = h->K * (fp8 ? 1 : 2), srow = h->K / 32;
  int64_t M = 0;
  const void* xs[kGatherMaxBlocks];
  const void* ss[kGatherMaxBlocks];
  int64_t xb[kGatherMaxBlocks], sb[kGatherMaxBlocks];
  for (int b = 0; b < nblocks; ++b) {
    const bi_gemm_block& k = blocks[b];
    if (k.rows < 0 || (k.rows > 0 && !k.x) || (fp8 && k.rows > 0 && !k.sx) || (!fp8 && k.sx))
      return BI_GEMM_ERR_INVALID_ARG;
    if (!is_aligned(k.x, 16) || (fp8 && !is_aligned(k.sx, 4))) return BI_GEMM_ERR_ALIGNMENT;
    M += k.rows;
    if (M >= (int64_t(1) << 31)) return BI_GEMM_ERR_UNSUPPORTED;
    xs[b] = k.x;
    ss[b] = k.sx;
    xb[b] = k.rows * xrow;
    sb[b] = k.rows * srow;
  }
  if (fp8 && (!sx_out || !sw)) return BI_GEMM_ERR_INVALID_ARG;
  if (!fp8 && (sx_out || sw)) return BI_GEMM_ERR_INVALID_ARG;
  if (M == 0) return BI_GEMM_OK;
  bi_gemm_scales sc{sx_out, sw};
  int rc = validate_run(h, x_out, M, W, fp8 ? &sc : nullptr, y);
  if (rc != BI_GEMM_OK) return rc;
  std::lock_guard<std::mutex> lk(h->mu);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = launch_gather(xs, xb, nblocks, x_out, 16, h->num_sms, st);
  if (rc == BI_GEMM_OK && fp8) rc = launch_gather(ss, sb, nblocks, sx_out, 4, h->num_sms, st);
  if (rc != BI_GEMM_OK) return rc;
  return launch(h, x_out, M, W, fp8 ? &sc : nullptr, y, st, 0, 0u);
}

BI_GEMM_API const char* bi_gemm_strerror(int code) {
  switch (code) {
    case BI_GEMM_OK: return "ok";
    case BI_GEMM_ERR_INVALID_ARG: return "invalid argument";
    case BI_GEMM_ERR_UNSUPPORTED: return "unsupported shape, dtype or device";
    case BI_GEMM_ERR_ALIGNMENT: return "pointer or row pitch not 16-byte aligned";
    case BI_GEMM_ERR_CUDA: return "CUDA runtime error";
    case BI_GEMM_ERR_OOM: return "workspace allocation failed";
    case BI_GEMM_ERR_TIMEOUT: return "bounded in-kernel wait expired";
    case BI_GEMM_ERR_SCRATCH_LIMIT: return "problem too large for the fixed scratch of bi_gemm_run_noalloc";
    default: return "unknown error code";
  }
}

BI_GEMM_API int bi_gemm_version(void) { return kVersion; }

#ifndef BI_GEMM_CONTROLS
// ------------------------------------------------------------------ allocation-free run
//
// bi_gemm_run grows a per-handle workspace with cudaMallocAsync when a split count S > 1 needs
// fp32 partials.  Some callers may not allocate device memory at call time: code whose device
// memory is entirely owned and budgeted by another framework's pool (a raw allocation there can
// fail or fragment it), latency-critical loops that must not take the allocator's locks or its
// implicit synchronisation, and code running where CUDA API allocation is not permitted.
// bi_gemm_run_noalloc gives them the same split-K kernel with its scratch (arrival counters and
// partials) in one fixed device array below, compiled into the library.
//
// The array is kNoAllocScratchBytes per device; every GPU on which this library's kernels are
// loaded holds it until the process exits.  Host code may not use the array's name as a device
// address (it is a host-side stand-in); the device address is fetched with cudaGetSymbolAddress,
// with the device current, by the first bi_gemm_run_noalloc call in each CUDA context, and kept
// with that context's unique id: a context created later (after cudaDeviceReset, say, where the
// module is loaded again and the array may sit elsewhere) gets its own lookup.

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;     // 8 MiB per device
// Arrival counters first.  The partials bound is the one that binds: the smallest partial
// block of a sub-tile (S = 2, BN = 64) is 64 KiB, so at most 127 sub-tiles fit beside the
// counters, far fewer than the 1024 counters these 4 KiB hold.
constexpr size_t kNoAllocCounterBytes = 4096;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct NoAllocSlot {
  unsigned long long ctx_id = 0;   // id of the context the address belongs to
  void* ptr = nullptr;
};
std::mutex g_noalloc_mu;
NoAllocSlot g_noalloc[kNoAllocMaxDevices];

// The current context's unique id (cuCtxGetId), or false when no context is current.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext c = nullptr;
  if (!get_cur || !get_id || get_cur(&c) != CUDA_SUCCESS || !c) return false;
  return get_id(c, id) == CUDA_SUCCESS;
}

int noalloc_scratch_address(int dev, char** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return BI_GEMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocSlot& slot = g_noalloc[dev];
  unsigned long long id = 0;
  const bool have_ctx = current_context_id(&id);
  if (!have_ctx || !slot.ptr || slot.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return BI_GEMM_ERR_CUDA;
    }
    // the lookup has made the device's context current if none was
    if (!current_context_id(&id)) return BI_GEMM_ERR_CUDA;
    slot.ptr = p;
    slot.ctx_id = id;
  }
  *out = static_cast<char*>(slot.ptr);
  return BI_GEMM_OK;
}

}  // namespace

BI_GEMM_API int bi_gemm_run_noalloc(bi_gemm_t h, const void* x, int64_t M, const void* W,
                                    const bi_gemm_scales* scales, void* y, void* stream) {
  int rc = validate_run(h, x, M, W, scales, y);
  if (rc != BI_GEMM_OK || M == 0) return rc;
  std::lock_guard<std::mutex> lk(h->mu);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BI_GEMM_ERR_CUDA;
  }
  if (dev != h->device) return BI_GEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int split = h->split;
  const Shape sh = shape_of(h, M);
  char* scratch = nullptr;
  if (split > 1) {
    const size_t part = size_t(sh.subtiles) * split * kBM * h->kern.bn * sizeof(float);
    if (size_t(sh.subtiles) * sizeof(uint32_t) > kNoAllocCounterBytes ||
        part > kNoAllocScratchBytes - kNoAllocCounterBytes)
      return BI_GEMM_ERR_SCRATCH_LIMIT;
    rc = noalloc_scratch_address(dev, &scratch);
    if (rc != BI_GEMM_OK) return rc;
    // The previous call's counters are normally back at zero, but an aborted run can leave
    // them set: clear the ones this call uses.  Partials need no clearing (written before read).
    if (cudaMemsetAsync(scratch, 0, size_t(sh.subtiles) * sizeof(uint32_t), st) != cudaSuccess) {
      cudaGetLastError();
      return BI_GEMM_ERR_CUDA;
    }
  }
  return launch_core(h, x, M, W, scales, y, st, split,
                     split > 1 ? reinterpret_cast<float*>(scratch + kNoAllocCounterBytes) : nullptr,
                     split > 1 ? reinterpret_cast<uint32_t*>(scratch) : nullptr, 0u);
}
#endif
