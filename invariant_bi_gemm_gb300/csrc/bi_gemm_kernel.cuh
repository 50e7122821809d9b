// bi_gemm_kernel.cuh — the batch-invariant GEMM kernel for sm_103a (TMA + tcgen05 + TMEM).
//
// y[M,N] = x[M,K] · W[K,N], fp32 accumulation, one compiled configuration per handle.
//
// Why this is batch invariant ("Batch-invariant matrix multiplication", nondeterminism
// article: the three breakers are M-dependent split-K, stream-K and a smaller tensor-core
// instruction at small M; the cure is one kernel configuration for every shape):
//   * the output tile is always 128 x BN (256 x BN on a CTA pair), the tcgen05 instruction
//     always M=128 (M=256 on a pair) x N=BN x K=16 (bf16) or K=32 (MXFP8), whatever M is;
//   * every output element is reduced over k-blocks kb = 0 .. KB-1 in ascending order, and
//     within a k-block over the same fixed sequence of MMA instructions;
//   * a split count S > 1 is fixed when the handle is created (from K, N and the SM count,
//     never M); split s always covers the same k-blocks, and the S fp32 partials of every
//     element are summed in the fixed serial order ((p0 + p1) + p2) + ..., whichever CTA does
//     the sum (integer arrival counters; no floating-point atomics);
//   * rows beyond M are zero-filled by TMA and never stored; a row's products never meet
//     another row's, so neither M nor the other rows' contents can reach row i.
// The persistent tile order (which SM computes which tile, and when) does change with M,
// but it decides no arithmetic: a tile's value is the same wherever it runs.  So does the
// pipeline's grouping on the pair tile (two k-blocks a stage when the x box has at most 64
// rows), which changes when the issuer waits, not which MMAs it issues or in what order.
//
// Tile = 128 x BN per CTA, or 256 x BN per CTA pair (CTAS = 2, BN = 256): the pair issues one
// tcgen05.mma.cta_group::2 of M=256, each CTA staging its own 128 rows of x and its own BN/2
// columns of W and receiving its 128 rows of the accumulator in its own TMEM.  For MXFP8 each
// CTA also stages its own rows' x scales and the scales of all BN columns of W, which the
// block-scaled pair MMA reads from each CTA's own TMEM.  The pair is one fixed configuration
// chosen from N, like everything else.
//
// Warp roles (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: x tile [128 x BK] (K-major, 128-byte swizzle) and W tile
//               [BK x BN] (N-major, 128-byte swizzle) per pipeline stage;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer;
//   warps 2-7   (MXFP8 only) scale producers, taking the k-blocks in turn: E8M0 scales into
//               the tcgen05.cp layout, then (leader CTA) tcgen05.cp into TMEM;
//   last 8      epilogue: tcgen05.ld -> round to nearest even -> TMA stores of 32 x 32 blocks,
//               or fp32 partials + ordered merge when S > 1.
// Every wait is bounded in time; on expiry the kernel records an error bit in the
// handle's status word, lets in-flight copies and MMAs finish, frees TMEM and returns.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace bigemm {

constexpr int kBM = 128;

// Error bits written to the status word (any non-zero value is reported as a timeout).
enum : uint32_t {
  kErrTimeoutProducer = 1u,
  kErrTimeoutMma = 2u,
  kErrTimeoutEpilogue = 4u,
  kErrTimeoutScales = 8u,
  kErrTimeoutMerge = 16u,
};

struct KParams {
  void* y;                  // [M, N] bf16 or fp32, row-major
  const uint8_t* sx;        // MXFP8: [M, K/32] E8M0
  const uint8_t* sw;        // MXFP8: [K/32, N] E8M0
  float* ws;                // split-K partials [tiles][S][128][BN] fp32 (S > 1)
  uint32_t* counters;       // split-K arrival counters [tiles] (S > 1)
  uint32_t* status;         // error word
  int32_t M, N, K;
  int32_t m_tiles, n_tiles;
  int32_t splits;           // S
  int32_t kblocks;          // KB = ceil(K / BK)
  int32_t a_box_rows;       // rows per x TMA box: 128, or round_up(M, 8) when M < 128
  int32_t group_n;          // raster order: N tiles per group (M tiles vary fastest within it)
  int32_t coop_merge;       // S > 1, every unit has its own resident CTA group and the merge is
                            // large: the S split CTAs of a sub-tile share it (else the last to
                            // arrive merges alone)
  int32_t w_early;          // W may be loaded before the previous kernel in the stream completes
  int32_t small_m;          // bf16 pair tile, x box of at most 64 rows: the small-M pipeline below
  int32_t small_stages;     // its stages (two k-blocks each)
  uint32_t slot_bytes;      // its k-block slot: the x box's rows, then the W tile
  uint64_t timeout_ns;
  uint32_t test_flags;      // only read by the control build
};

constexpr __host__ __device__ int pow2_ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <bool kFp8_, bool kOutF32_, int kBN_, int kStages_, int kAccBufs_, int kCtas_ = 1>
struct KCfg {
  static constexpr bool kFp8 = kFp8_;
  static constexpr bool kOutF32 = kOutF32_;
  static constexpr int BN = kBN_;
  static constexpr int STAGES = kStages_;
  static constexpr int ACC_BUFS = kAccBufs_;
  static constexpr int CTAS = kCtas_;                   // CTAs per output tile (1 or 2)
  static_assert(CTAS == 1 || (CTAS == 2 && (kBN_ == 256 || (!kFp8_ && kBN_ == 192))),
                "CTA pairs: BN = 256 (bf16 or MXFP8) or 192 (bf16)");
  static constexpr int TILE_M = kBM * CTAS;
  static constexpr int BN_CTA = BN / CTAS;              // W columns staged by each CTA
  static constexpr int ELEM = kFp8 ? 1 : 2;
  static constexpr int BK = 128 / ELEM;                 // one 128-byte swizzle row of K
  static constexpr int MMA_K = kFp8 ? 32 : 16;          // K per tcgen05.mma
  static constexpr int K_STEPS = BK / MMA_K;            // 4
  // W is staged N-major in 128-byte swizzle atoms (64 bf16 / 128 E4M3 columns), or 64-byte
  // atoms (32 bf16 columns) when a CTA's share of the tile is not a multiple of 64 columns.
  static constexpr int B_SW = (BN_CTA * ELEM) % 128 == 0 ? 128 : 64;   // swizzle span in bytes
  static constexpr int ATOM_N = B_SW / ELEM;             // N per swizzle row of W
  static constexpr int N_ATOMS = BN_CTA / ATOM_N;        // swizzle atoms of W per CTA
  static_assert(BN_CTA % ATOM_N == 0 && BN >= 16 && BN <= 256, "BN");
  static constexpr uint32_t B_LAYOUT = B_SW == 128 ? 2u : 4u;   // descriptor layout code
  static constexpr int A_BYTES = kBM * 128;             // 16 KB
  static constexpr int B_ATOM_BYTES = BK * B_SW;
  static constexpr int B_BYTES = N_ATOMS * B_ATOM_BYTES;
  // Small-M pipeline (bf16 pair tile, x box of at most 64 rows): the same ring holds stages of
  // two k-blocks, each k-block a slot of the x box's rows followed by its W tile, so that the MMA
  // issuer waits once per eight MMAs and more bytes are in flight than six full stages allow.
  // The instructions, their operands and their order are those of the other pipeline.
  static constexpr bool SMALLM = !kFp8 && CTAS == 2;
  static constexpr int RING_BYTES = STAGES * (A_BYTES + B_BYTES);
  static constexpr int SFA_BYTES = kFp8 ? 512 : 0;      // 128 rows x 4 k-blocks
  // Each CTA stages the scales of all BN columns: on a pair, the block-scaled MMA reads the B
  // scales of the whole N extent from each CTA's own TMEM.
  static constexpr int SFB_BYTES = kFp8 ? (BN / 128) * 512 : 0;
  static constexpr int SF_BYTES = SFA_BYTES + SFB_BYTES;
  static constexpr int EPI_WARPS = 8;                   // two per TMEM lane quarter
  // MXFP8: six scale-producer warps take the k-blocks in turn, so that the load latency of six
  // stages' scales overlaps.
  static constexpr int SCALE_WARPS = kFp8 ? 6 : 0;
  // Each scale warp owns one stage's scale slot (warp j fills items j, j + STAGES, ...), so a
  // warp's wait for the slot's previous copy (a parity wait on sfdone_bar) can never see a phase
  // two behind; with more scale warps than stages two warps would share a slot and that wait
  // could pass on the wrong phase.
  static_assert(!kFp8 || SCALE_WARPS == STAGES, "MXFP8: one scale warp per stage");
  static constexpr int NUM_WARPS = 2 + SCALE_WARPS + EPI_WARPS;
  static constexpr int EPI_WARP0 = NUM_WARPS - EPI_WARPS;
  // MXFP8 kernels launch 16 warps (128 registers a thread); setmaxnreg then moves registers from
  // the two producer warpgroups (TMA, MMA, scales) to the two epilogue warpgroups.
  static constexpr bool kRegSplit = kFp8;
  // (the single-accumulator epilogue holds a warp's whole share of the tile in registers)
  static constexpr int REGS_LOW = ACC_BUFS == 1 ? 64 : 80;
  static constexpr int REGS_HIGH = ACC_BUFS == 1 ? 192 : 176;
  static_assert(!kRegSplit || (NUM_WARPS == 16 && EPI_WARP0 == 8), "register split: whole warpgroups");
  static_assert(!kRegSplit || EPI_WARP0 * 32 * REGS_LOW + EPI_WARPS * 32 * REGS_HIGH <= 65536,
                "register split exceeds the launch's registers");
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = NUM_WARPS * 32;
  // TMEM columns: accumulators first, then 16 columns of scale factors per stage.
  static constexpr int SF_TMEM_COL0 = ACC_BUFS * BN;
  static constexpr int TMEM_USED = SF_TMEM_COL0 + (kFp8 ? 16 * STAGES : 0);
  static constexpr int TMEM_COLS = pow2_ceil(TMEM_USED < 32 ? 32 : TMEM_USED);
  static_assert(TMEM_COLS <= 512, "TMEM");
  // shared memory offsets from a 1024-byte aligned base
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_SF + STAGES * SF_BYTES;
  // full, empty, accumulator full / empty, drain, epilogue; MXFP8 adds per stage the peer's
  // scales-ready barrier and per scale warp a drain barrier for its scale copies
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 2 + (kFp8 ? 2 * STAGES + SCALE_WARPS : 0);
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // epilogue staging for TMA stores: per epilogue warp, one or two 32 x 32 output blocks
  static constexpr int OUT_BYTES = kOutF32 ? 4 : 2;
  static constexpr int STG_BYTES = 32 * 32 * OUT_BYTES;
  static constexpr int OFF_STG = (OFF_MISC + 16 + 1023) / 1024 * 1024;   // swizzle-atom aligned
  static constexpr int STG_BUFS =
      OFF_STG + EPI_WARPS * 2 * STG_BYTES + 1024 <= 232448 ? 2 : 1;
  static constexpr int SMEM_BYTES = OFF_STG + EPI_WARPS * STG_BUFS * STG_BYTES + 1024;  // + slack
  static_assert(SMEM_BYTES <= 232448, "shared memory");

  // tcgen05 instruction descriptor (kind::f16): D=f32, A=B=bf16, A K-major, B N-major.
  static constexpr uint32_t IDESC_BF16 =
      (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
      (uint32_t(BN >> 3) << 17) | (uint32_t(TILE_M >> 4) << 24);
  // tcgen05 instruction descriptor (kind::mxf8f6f4 block-scaled): A=B=E4M3, A K-major,
  // B N-major, E8M0 scales; the scale-factor byte selectors are OR-ed in per K step.
  static constexpr uint32_t IDESC_MXF8 =
      (0u << 7) | (0u << 10) | (0u << 15) | (1u << 16) | (uint32_t(BN >> 3) << 17) |
      (1u << 23) | (uint32_t(TILE_M >> 4) << 24);
};

// Shared-memory matrix descriptor: start, leading / stride byte offsets, version 1, layout.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t layout) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (uint64_t(layout) << 61);
}
constexpr uint32_t kLayoutNone = 0;
constexpr uint32_t kLayoutSW128 = 2;

struct SyncCtx {
  volatile uint32_t* abort;  // shared: set once any role gives up
  uint32_t* status;          // global error word
  uint64_t timeout_ns;
};

// Bounded wait on an mbarrier phase.  Returns false (and raises the abort flag and the error
// bit) once the time limit passes, or as soon as another role has aborted.
// How a wait observes a barrier phase: acquire at CTA scope (default) or acquire at cluster
// scope (the phase completes with arrivals from the peer CTA).
enum class Wait { kCta, kCluster };

template <Wait kW = Wait::kCta>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  if constexpr (kW == Wait::kCluster)
    return ptx::mbar_try_wait_cluster(bar, parity);
  else
    return ptx::mbar_try_wait(bar, parity);
}

template <Wait kW = Wait::kCta>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const SyncCtx& c,
                                           uint32_t err_bit) {
  if (try_wait<kW>(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (try_wait<kW>(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*c.abort) return false;
      if (ptx::globaltimer() - t0 > c.timeout_ns) {
        *c.abort = 1u;
        atomicOr(c.status, err_bit);
        return false;
      }
    }
  }
}

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast, and on success every
// lane observes the (already completed) phase itself before touching the guarded data.
template <Wait kW = Wait::kCta>
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, const SyncCtx& c,
                                                uint32_t err_bit) {
  const int lane = threadIdx.x & 31;
  uint32_t ok = 1;
  if (lane == 0) ok = wait_phase<kW>(bar, parity, c, err_bit) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) {
    for (int i = 0; i < (1 << 20) && !try_wait<kW>(bar, parity); ++i) {
    }
  }
  return ok != 0;
}

struct UnitCoord {
  int tile, s, m_tile, n_tile, kb_begin, kb_end;
};

// Unit u -> output tile and split s.  Tiles are visited in groups of group_n N-tiles; within a
// group the N tile varies fastest and the M tile slowest, so the tiles resident at one time
// share a few x row blocks and a few W column slabs (L2 reuse).  The order decides no
// arithmetic.  Split s covers k-blocks [s*q + min(s, r), (s+1)*q + min(s+1, r)) with
// q = KB / S, r = KB % S (fixed by K and S).
__device__ __forceinline__ UnitCoord unit_coord(int u, const KParams& p) {
  UnitCoord c;
  if (p.splits == 1) {
    c.tile = u;
    c.s = 0;
    c.kb_begin = 0;
    c.kb_end = p.kblocks;
  } else {
    c.tile = u / p.splits;
    c.s = u - c.tile * p.splits;
    const int q = p.kblocks / p.splits, r = p.kblocks - q * p.splits;
    c.kb_begin = c.s * q + min(c.s, r);
    c.kb_end = c.kb_begin + q + (c.s < r ? 1 : 0);
  }
  const int per_group = p.group_n * p.m_tiles;
  const int g = c.tile / per_group;
  const int local = c.tile - g * per_group;
  const int gn = min(p.group_n, p.n_tiles - g * p.group_n);   // N tiles in this (last) group
  c.m_tile = local / gn;
  c.n_tile = g * p.group_n + (local - c.m_tile * gn);
  return c;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    bi_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_y, const KParams p) {
  constexpr bool kPair = C::CTAS == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + C::ACC_BUFS + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 2 * C::ACC_BUFS);
  const uint32_t epi_bar = drain_bar + 8u;   // split-K hand-off among the epilogue warps
  // MXFP8: the peer CTA's scales for a stage are in its shared memory (pairs only)
  auto sfpeer_bar = [&](int s) { return epi_bar + 8u + 8u * s; };
  // MXFP8: completion of a scale warp's last scale copies
  auto sfdrain_bar = [&](int w) { return epi_bar + 8u + 8u * (C::STAGES + w); };
  // MXFP8: a stage's scale slot has been copied into TMEM (in both CTAs of a pair) and may be
  // refilled
  auto sfdone_bar = [&](int s) { return epi_bar + 8u + 8u * (C::STAGES + C::SCALE_WARPS + s); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  uint32_t* tmem_slot = misc + 0;
  volatile uint32_t* abort_flag = misc + 1;
  volatile uint32_t* last_flag = misc + 2;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? ptx::cluster_ctarank() : 0u;   // 0 = leader (issues the MMAs)
  const int group = blockIdx.x / C::CTAS;                        // this CTA's tile group
  const int ngroups = gridDim.x / C::CTAS;
  const int units = p.m_tiles * p.n_tiles * p.splits;

  if (warp == C::EPI_WARP0) {
    // An idle warp touches the scalar parameters first, so that their constant-cache line is
    // resident by the time the producer computes its first tile.
    asm volatile("" ::"r"(p.M), "r"(p.N), "r"(p.K), "r"(p.m_tiles), "r"(p.n_tiles), "r"(p.splits),
                 "r"(p.kblocks), "r"(p.a_box_rows));
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // TMA bytes (+ the commit of the stage's scale copies, MXFP8)
      ptx::mbar_init(full_bar(s), C::kFp8 ? 2u : 1u);
      ptx::mbar_init(empty_bar(s), 1u);
    }
    for (int b = 0; b < C::ACC_BUFS; ++b) {
      ptx::mbar_init(tfull_bar(b), 1u);
      ptx::mbar_init(tempty_bar(b), uint32_t(C::EPI_WARPS * C::CTAS));
    }
    ptx::mbar_init(drain_bar, 1u);
    ptx::mbar_init(epi_bar, uint32_t(C::EPI_WARPS));
    if constexpr (C::kFp8) {
      for (int s = 0; s < C::STAGES; ++s) ptx::mbar_init(sfpeer_bar(s), 1u);
      for (int w = 0; w < C::SCALE_WARPS; ++w) ptx::mbar_init(sfdrain_bar(w), 1u);
      for (int s = 0; s < C::STAGES; ++s) ptx::mbar_init(sfdone_bar(s), 1u);
    }
    *abort_flag = 0u;
    *last_flag = 0u;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::prefetch_tensormap(&tmap_x);
    ptx::prefetch_tensormap(&tmap_w);
    ptx::prefetch_tensormap(&tmap_y);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  // Pairs: announce "barriers initialised, TMEM allocated" to the peer now, and wait for the
  // peer's announcement only where it matters (before touching the peer's barriers or TMEM).
  if constexpr (kPair) ptx::cluster_arrive();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const SyncCtx sc{abort_flag, p.status, p.timeout_ns};
  // Set-up touches only this CTA's shared memory and TMEM, so it may overlap the tail of the
  // previous kernel in the stream.  Each role waits for that kernel to complete
  // (grid_dependency_wait) just before its first global-memory access.

  if (warp < C::EPI_WARP0) {
    // producer warpgroups: TMA, MMA issue (and MXFP8 scales) need few registers
    if constexpr (C::kRegSplit) ptx::setmaxnreg_dec<C::REGS_LOW>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if constexpr (kPair) {
        if (lane != 0 || rank != 0) ptx::cluster_wait();   // the peer signals the leader's barriers
      }
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_par = 0;   // per stage: an issue is outstanding / its parity
        bool ok = true;
        // Issue the loads of one k-block into stage `st`: with `w_part` the stage's byte count and
        // the W tiles, with `x_part` the x tile.
        auto issue = [&](int st, const UnitCoord& uc, int kb, bool w_part, bool x_part) {
          const uint32_t fb = full_bar(st);
          const uint32_t adst = sbase + C::OFF_A + st * C::A_BYTES;
          const uint32_t bdst = sbase + C::OFF_B + st * C::B_BYTES;
          const int row0 = uc.m_tile * C::TILE_M + int(rank) * kBM;
          const int col0 = uc.n_tile * C::BN + int(rank) * C::BN_CTA;
          // x rows at or past M are never stored, so they need not be loaded: a CTA whose 128
          // rows all lie past M skips its x tile, and the x box is only as tall as M needs.
          // The shared-memory rows left unwritten feed only those discarded output rows.
          const uint32_t a_bytes = uint32_t(p.a_box_rows) * 128u;
          const bool load_a = row0 < p.M;
          if constexpr (kPair) {
            const uint32_t lfb = ptx::mapa_shared(fb, 0);   // the leader's full barrier
            if (w_part && rank == 0) {
              const bool peer_a = row0 + kBM < p.M;
              ptx::mbar_arrive_expect_tx(fb, (load_a ? a_bytes : 0u) + (peer_a ? a_bytes : 0u) +
                                                 uint32_t(C::CTAS * C::B_BYTES));
            }
            if (x_part && load_a) ptx::tma_load_2d_pair(adst, &tmap_x, lfb, kb * C::BK, row0);
            if (w_part) {
  #pragma unroll
              for (int a = 0; a < C::N_ATOMS; ++a)
                ptx::tma_load_2d_pair(bdst + a * C::B_ATOM_BYTES, &tmap_w, lfb, col0 + a * C::ATOM_N,
                                      kb * C::BK);
            }
          } else {
            if (w_part) ptx::mbar_arrive_expect_tx(fb, a_bytes + uint32_t(C::B_BYTES));
            if (x_part) ptx::tma_load_2d(adst, &tmap_x, fb, kb * C::BK, row0);
            if (w_part) {
  #pragma unroll
              for (int a = 0; a < C::N_ATOMS; ++a)
                ptx::tma_load_2d(bdst + a * C::B_ATOM_BYTES, &tmap_w, fb, col0 + a * C::ATOM_N, kb * C::BK);
            }
          }
          issued_mask |= 1u << st;
          issued_par = (issued_par & ~(1u << st)) | (phase << st);
        };
        bool small_done = false;
        if constexpr (C::SMALLM) {
         if (p.small_m) {
          // Small-M pipeline: stage st holds k-blocks kb, kb + 1 in slots 2st, 2st + 1, each the
          // x box's rows followed by the W tile; otherwise as below.
          const int nst = p.small_stages;
          const uint32_t a_bytes = uint32_t(p.a_box_rows) * 128u;
          auto issue2 = [&](int st, const UnitCoord& uc, int kb, int nsub, bool w_part, bool x_part) {
            const uint32_t fb = full_bar(st);
            const uint32_t lfb = ptx::mapa_shared(fb, 0);   // the leader's full barrier
            const int row0 = uc.m_tile * C::TILE_M + int(rank) * kBM;
            const int col0 = uc.n_tile * C::BN + int(rank) * C::BN_CTA;
            const bool load_a = row0 < p.M;              // (the peer's rows all lie past M here)
            if (w_part && rank == 0)
              ptx::mbar_arrive_expect_tx(fb, uint32_t(nsub) * ((load_a ? a_bytes : 0u) + uint32_t(C::CTAS * C::B_BYTES)));
  #pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (j < nsub) {
                const uint32_t adst = sbase + uint32_t(st * 2 + j) * p.slot_bytes;
                const uint32_t bdst = adst + p.slot_bytes - uint32_t(C::B_BYTES);
                const int kc = (kb + j) * C::BK;
                if (x_part && load_a) ptx::tma_load_2d_pair(adst, &tmap_x, lfb, kc, row0);
                if (w_part) {
  #pragma unroll
                  for (int a = 0; a < C::N_ATOMS; ++a)
                    ptx::tma_load_2d_pair(bdst + a * C::B_ATOM_BYTES, &tmap_w, lfb, col0 + a * C::ATOM_N, kc);
                }
              }
            }
            issued_mask |= 1u << st;
            issued_par = (issued_par & ~(1u << st)) | (phase << st);
          };
          int pre = 0;
          bool early = p.w_early != 0;
  #ifdef BI_GEMM_CONTROLS
          early = early && !(p.test_flags & 1u);
  #endif
          if (early) {
            for (int u = group; u < units && pre < nst; u += ngroups) {
              const UnitCoord uc = unit_coord(u, p);
              for (int kb = uc.kb_begin; kb < uc.kb_end && pre < nst; kb += 2, ++pre)
                issue2(pre, uc, kb, min(2, uc.kb_end - kb), true, false);
            }
          }
          ptx::grid_dependency_wait();
          int item = 0;
          for (int u = group; u < units && ok; u += ngroups) {
            const UnitCoord uc = unit_coord(u, p);
            for (int kb = uc.kb_begin; kb < uc.kb_end; kb += 2, ++item) {
              const int nsub = min(2, uc.kb_end - kb);
              if (item < pre) {
                issue2(stage, uc, kb, nsub, false, true);
              } else {
                if (!wait_phase(empty_bar(stage), phase ^ 1u, sc, kErrTimeoutProducer)) {
                  ok = false;
                  break;
                }
                bool skip = false;
  #ifdef BI_GEMM_CONTROLS
                skip = (p.test_flags & 1u) && u == group && kb == uc.kb_begin;
  #endif
                if (!skip) issue2(stage, uc, kb, nsub, true, true);
              }
              if (++stage == nst) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
          small_done = true;
         }
        }
        if (!small_done) {
          // W is only read.  When the caller has declared that no kernel which may still be running
          // writes it (p.w_early), the W tiles of this CTA's first STAGES k-blocks are issued before
          // the wait for the previous kernel in the stream; only x (which may be that kernel's
          // output) and every later load wait for it.  The stages are fresh, so no empty-barrier
          // wait is needed for them.
          int pre = 0;
          bool early = p.w_early != 0;
    #ifdef BI_GEMM_CONTROLS
          early = early && !(p.test_flags & 1u);
    #endif
          if (early) {
            for (int u = group; u < units && pre < C::STAGES; u += ngroups) {
              const UnitCoord uc = unit_coord(u, p);
              for (int kb = uc.kb_begin; kb < uc.kb_end && pre < C::STAGES; ++kb, ++pre)
                issue(pre, uc, kb, true, false);
            }
          }
          ptx::grid_dependency_wait();
          int item = 0;
          for (int u = group; u < units && ok; u += ngroups) {
            const UnitCoord uc = unit_coord(u, p);
            for (int kb = uc.kb_begin; kb < uc.kb_end; ++kb, ++item) {
              if (item < pre) {
                issue(stage, uc, kb, false, true);          // its W is already on the way
              } else {
                if (!wait_phase(empty_bar(stage), phase ^ 1u, sc, kErrTimeoutProducer)) {
                  ok = false;
                  break;
                }
                bool skip = false;
    #ifdef BI_GEMM_CONTROLS
                // control build only: withhold one stage so that the consumer's bounded wait expires
                skip = (p.test_flags & 1u) && u == group && kb == uc.kb_begin;
    #endif
                if (!skip) issue(stage, uc, kb, true, true);
              }
              if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        }
        ptx::launch_dependents();   // this CTA has issued all its loads
        if constexpr (kPair) {
          if (rank == 0) ptx::cluster_wait();
        }
        if (!ok) {
          // let every copy already in flight land before the CTA can exit
          if (rank == 0) {
            SyncCtx drain{abort_flag, p.status, p.timeout_ns};
            volatile uint32_t no_abort = 0;
            drain.abort = &no_abort;
            for (int s = 0; s < C::STAGES; ++s)
              if (issued_mask & (1u << s))
                wait_phase(full_bar(s), (issued_par >> s) & 1u, drain, kErrTimeoutProducer);
          } else if (issued_mask) {
            // the peer's copies are counted on the leader's barriers: give them time to land
            const uint64_t t0 = ptx::globaltimer();
            while (ptx::globaltimer() - t0 < 2000000ull) {
            }
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer (leader CTA)
      if constexpr (kPair) ptx::cluster_wait();            // the peer's TMEM is allocated
      if (lane == 0 && rank == 0) {
        int stage = 0;
        uint32_t phase = 0;
        int buf = 0;
        uint32_t bphase = 0;
        bool ok = true, issued_any = false;
        bool small_done = false;
        if constexpr (C::SMALLM) {
         if (p.small_m) {
          // Small-M pipeline (see the producer): one wait and one commit per two k-blocks, the
          // same MMAs in the same order as below.
          const int nst = p.small_stages;
          for (int u = group; u < units && ok; u += ngroups) {
            const UnitCoord uc = unit_coord(u, p);
            if (!wait_phase(tempty_bar(buf), bphase ^ 1u, sc, kErrTimeoutMma)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + uint32_t(buf * C::BN);
            for (int kb = uc.kb_begin; kb < uc.kb_end; kb += 2) {
              if (!wait_phase(full_bar(stage), phase, sc, kErrTimeoutMma)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              const int nsub = min(2, uc.kb_end - kb);
  #pragma unroll
              for (int j = 0; j < 2; ++j) {
                if (j < nsub) {
                  const uint32_t a_addr = sbase + uint32_t(stage * 2 + j) * p.slot_bytes;
                  const uint32_t b_addr = a_addr + p.slot_bytes - uint32_t(C::B_BYTES);
  #pragma unroll
                  for (int kk = 0; kk < C::K_STEPS; ++kk) {
                    const uint64_t ad = make_sdesc(a_addr + kk * 32, 16, 1024, kLayoutSW128);
                    const uint64_t bd = make_sdesc(b_addr + kk * C::MMA_K * C::B_SW, C::B_ATOM_BYTES,
                                                   8 * C::B_SW, C::B_LAYOUT);
                    const uint32_t acc = (kb + j != uc.kb_begin || kk != 0) ? 1u : 0u;
                    ptx::mma_bf16_pair(d_tmem, ad, bd, C::IDESC_BF16, acc);
                  }
                }
              }
              issued_any = true;
              ptx::tc_commit_pair_mc(empty_bar(stage), 0x3);   // frees the stage in both CTAs
              if (++stage == nst) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            ptx::tc_commit_pair_mc(tfull_bar(buf), 0x3);       // both CTAs' epilogues
            if (++buf == C::ACC_BUFS) {
              buf = 0;
              bphase ^= 1u;
            }
          }
          small_done = true;
         }
        }
        if (!small_done) {
          for (int u = group; u < units && ok; u += ngroups) {
            const UnitCoord uc = unit_coord(u, p);
            if (!wait_phase(tempty_bar(buf), bphase ^ 1u, sc, kErrTimeoutMma)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + uint32_t(buf * C::BN);
            for (int kb = uc.kb_begin; kb < uc.kb_end; ++kb) {
              if (!wait_phase(full_bar(stage), phase, sc, kErrTimeoutMma)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              const uint32_t a_addr = sbase + C::OFF_A + stage * C::A_BYTES;
              const uint32_t b_addr = sbase + C::OFF_B + stage * C::B_BYTES;
              if constexpr (C::kFp8) {
                // the stage's scales are already in TMEM: their copies were committed to full_bar
                const uint32_t sfa_t = tmem_base + uint32_t(C::SF_TMEM_COL0 + 16 * stage);
                const uint32_t sfb_t = sfa_t + 8u;
    #pragma unroll
                for (int kk = 0; kk < C::K_STEPS; ++kk) {
                  const uint64_t ad = make_sdesc(a_addr + kk * 32, 16, 1024, kLayoutSW128);
                  const uint64_t bd = make_sdesc(b_addr + kk * C::MMA_K * C::B_SW, C::B_ATOM_BYTES,
                                                 8 * C::B_SW, C::B_LAYOUT);
                  const uint32_t idesc = C::IDESC_MXF8 | (uint32_t(kk) << 4) | (uint32_t(kk) << 29);
                  const uint32_t acc = (kb != uc.kb_begin || kk != 0) ? 1u : 0u;
                  if constexpr (kPair)
                    ptx::mma_mxf8_pair(d_tmem, ad, bd, idesc, sfa_t, sfb_t, acc);
                  else
                    ptx::mma_mxf8(d_tmem, ad, bd, idesc, sfa_t, sfb_t, acc);
                }
              } else {
    #pragma unroll
                for (int kk = 0; kk < C::K_STEPS; ++kk) {
                  const uint64_t ad = make_sdesc(a_addr + kk * 32, 16, 1024, kLayoutSW128);
                  const uint64_t bd = make_sdesc(b_addr + kk * C::MMA_K * C::B_SW, C::B_ATOM_BYTES,
                                                 8 * C::B_SW, C::B_LAYOUT);
                  const uint32_t acc = (kb != uc.kb_begin || kk != 0) ? 1u : 0u;
                  if constexpr (kPair)
                    ptx::mma_bf16_pair(d_tmem, ad, bd, C::IDESC_BF16, acc);
                  else
                    ptx::mma_bf16(d_tmem, ad, bd, C::IDESC_BF16, acc);
                }
              }
              issued_any = true;
              if constexpr (kPair)
                ptx::tc_commit_pair_mc(empty_bar(stage), 0x3);   // frees the stage in both CTAs
              else
                ptx::tc_commit(empty_bar(stage));
              if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            if constexpr (kPair)
              ptx::tc_commit_pair_mc(tfull_bar(buf), 0x3);       // both CTAs' epilogues
            else
              ptx::tc_commit(tfull_bar(buf));
            if (++buf == C::ACC_BUFS) {
              buf = 0;
              bphase ^= 1u;
            }
          }
        }
        if (!ok && issued_any) {
          // wait for the MMAs already issued before TMEM is released
          if constexpr (kPair)
            ptx::tc_commit_pair_mc(drain_bar, 0x1);
          else
            ptx::tc_commit(drain_bar);
          SyncCtx drain{abort_flag, p.status, p.timeout_ns};
          volatile uint32_t no_abort = 0;
          drain.abort = &no_abort;
          wait_phase(drain_bar, 0u, drain, kErrTimeoutMma);
        }
      }
      __syncwarp();
    } else if (C::kFp8 && warp < 2 + C::SCALE_WARPS) {
      if constexpr (C::kFp8) {
        // ---------------------------------------------------------- scale producers (MXFP8)
        if constexpr (kPair) ptx::cluster_wait();
        // Layout expected by tcgen05.cp 32x128b.warpx4 for 128 rows x 4 k-blocks (512 bytes):
        // byte (r % 32) * 16 + (r / 32) * 4 + kblk.  One 512-byte block for this CTA's 128 rows
        // of x, one per 128 columns of the tile's W columns (all BN of them, on a pair too).
        // This CTA's k-block items are numbered it = 0, 1, ... in pipeline order; scale warp j
        // fills items j, j + SCALE_WARPS, ...: once the stage's scale slot has been copied into
        // TMEM for the previous item (sfdone_bar), it copies the item's scales into the slot
        // (cp.async) and rearranges them there, ahead of the MMAs.
        // On a pair the peer's warp publishes its slot to the leader (sfpeer_bar); the leader's
        // warp waits until the stage is free (its MMAs done), issues the tcgen05.cp of both CTAs'
        // scales and commits them to the stage's full barrier and to both CTAs' sfdone_bar, so
        // the MMA issuer finds the scales in TMEM and issues only MMAs.
        const int sw_id = warp - 2;
        const int KB32 = p.K / 32;
        int u = group, kb = 0, kb_end = 0, row_base = 0, col_base = 0;
        auto enter_unit = [&]() {
          const UnitCoord uc = unit_coord(u, p);
          kb = uc.kb_begin;
          kb_end = uc.kb_end;
          row_base = uc.m_tile * C::TILE_M + int(rank) * kBM;
          col_base = uc.n_tile * C::BN;
        };
        // step to the next item; false once this CTA has none left
        auto advance = [&]() -> bool {
          ++kb;
          while (kb >= kb_end) {
            u += ngroups;
            if (u >= units) return false;
            enter_unit();
          }
          return true;
        };
        constexpr int kChunksPerRow = C::BN / 16;                   // 16-byte chunks per W scale row
        ptx::grid_dependency_wait();
        bool ok = true, copied = false;   // lane 0: no wait gave up / issued scale copies
        bool valid = u < units;
        if (valid) enter_unit();
        for (int i = 0; i < sw_id && valid; ++i) valid = advance();
        int it = sw_id;
        while (valid) {
          const int stage = it % C::STAGES;
          const uint32_t phase = uint32_t(it / C::STAGES) & 1u;
          // The slot may be refilled once its previous scales are in TMEM: the loads and the
          // rearrangement below run up to STAGES items ahead of the MMAs; only the copy into
          // the stage's TMEM columns waits for the stage to be free.
          if (!warp_wait_phase(sfdone_bar(stage), phase ^ 1u, sc, kErrTimeoutScales)) break;
          const uint32_t sf_addr = sbase + C::OFF_SF + stage * C::SF_BYTES;
          const uint32_t sfb_addr = sf_addr + C::SFA_BYTES;
          // x: this k-block's four scales of a row (one 32-bit word) go straight to the row's place
          // in the layout; rows at or past M are zero-filled (their outputs are never stored)
  #pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int r = g * 32 + lane;
            const int row = row_base + r;
            const bool in = row < p.M;
            ptx::cp_async_4(sf_addr + uint32_t((r & 31) * 16 + (r >> 5) * 4),
                            in ? p.sx + (size_t)row * KB32 + 4 * kb : p.sx, in ? 4u : 0u);
          }
          // W: the four scale rows of this k-block over the tile's BN columns, as stored (4 rows x
          // BN bytes), in 16-byte chunks; columns at or past N (whole chunks, N % 16 == 0) are
          // zero-filled (never stored)
  #pragma unroll
          for (int i = 0; i < C::BN / 128; ++i) {
            const int c = i * 32 + lane;
            const int t = c / kChunksPerRow, cc = c - t * kChunksPerRow;
            const int col = col_base + cc * 16;
            const bool in = col < p.N;
            ptx::cp_async_16(sfb_addr + uint32_t(t * C::BN + cc * 16),
                             in ? p.sw + (size_t)(kb * 4 + t) * p.N + col : p.sw, in ? 16u : 0u);
          }
          ptx::cp_async_commit();
          ptx::cp_async_wait<0>();
          __syncwarp();                    // every lane's copies have landed
          // W scales, in place: lane l reads columns 4l .. 4l+3 of each scale row of each
          // 128-column block; a 4 x 4 byte transpose gives v[b][j], the four k-block scales of
          // column 4l + j; all reads precede all writes
          uint32_t v[C::BN / 128][4];
  #pragma unroll
          for (int b = 0; b < C::BN / 128; ++b) {
            uint32_t w[4];
  #pragma unroll
            for (int t = 0; t < 4; ++t) w[t] = ptx::ld_shared_u32(sfb_addr + t * C::BN + b * 128 + 4 * lane);
            const uint32_t lo01 = __byte_perm(w[0], w[1], 0x5140);
            const uint32_t hi01 = __byte_perm(w[0], w[1], 0x7362);
            const uint32_t lo23 = __byte_perm(w[2], w[3], 0x5140);
            const uint32_t hi23 = __byte_perm(w[2], w[3], 0x7362);
            v[b][0] = __byte_perm(lo01, lo23, 0x5410);
            v[b][1] = __byte_perm(lo01, lo23, 0x7632);
            v[b][2] = __byte_perm(hi01, hi23, 0x5410);
            v[b][3] = __byte_perm(hi01, hi23, 0x7632);
          }
          __syncwarp();
  #pragma unroll
          for (int b = 0; b < C::BN / 128; ++b) {
  #pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = 4 * lane + j;                    // column within this 128-column block
              ptx::st_shared_u32(sfb_addr + b * 512 + (c & 31) * 16 + (c >> 5) * 4, v[b][j]);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (kPair && rank != 0) {
              // peer: publish this stage's scales to the leader, which copies them into TMEM
              ptx::fence_release_shared();
              ptx::mbar_arrive_remote_relaxed(ptx::mapa_shared(sfpeer_bar(stage), 0));
            } else {
              // leader (or single CTA): once the peer's scales are in place too, copy both CTAs'
              // scales into TMEM and count the copies' completion on the stage's full barrier
              bool ready = wait_phase(empty_bar(stage), phase ^ 1u, sc, kErrTimeoutScales);
              if constexpr (kPair)
                ready = ready && wait_phase<Wait::kCluster>(sfpeer_bar(stage), phase, sc, kErrTimeoutScales);
              if (ready) {
                ptx::tc_fence_after();
                const uint32_t sfa_t = tmem_base + uint32_t(C::SF_TMEM_COL0 + 16 * stage);
                const uint32_t sfb_t = sfa_t + 8u;
                const uint64_t sfa_d = make_sdesc(sf_addr, 0, 128, kLayoutNone);
                if constexpr (kPair)
                  ptx::tc_cp_32x128b_x4_pair(sfa_t, sfa_d);
                else
                  ptx::tc_cp_32x128b_x4(sfa_t, sfa_d);
  #pragma unroll
                for (int b = 0; b < C::BN / 128; ++b) {
                  const uint64_t sfb_d = make_sdesc(sf_addr + C::SFA_BYTES + 512 * b, 0, 128, kLayoutNone);
                  if constexpr (kPair)
                    ptx::tc_cp_32x128b_x4_pair(sfb_t + 4u * b, sfb_d);
                  else
                    ptx::tc_cp_32x128b_x4(sfb_t + 4u * b, sfb_d);
                }
                if constexpr (kPair) {
                  ptx::tc_commit_pair_mc(full_bar(stage), 0x1);
                  ptx::tc_commit_pair_mc(sfdone_bar(stage), 0x3);   // both CTAs' slots are free
                } else {
                  ptx::tc_commit(full_bar(stage));
                  ptx::tc_commit(sfdone_bar(stage));
                }
                copied = true;
              }
              ok = ready;
            }
          }
          if (!__shfl_sync(0xffffffffu, ok ? 1u : 0u, 0)) break;
          for (int i = 0; i < C::SCALE_WARPS && valid; ++i) valid = advance();
          it += C::SCALE_WARPS;
        }
        ptx::cp_async_wait<0>();   // no copy may still target shared memory when the CTA exits
        // the last scale copies must land before the CTA may release TMEM
        if (lane == 0 && copied) {
          if constexpr (kPair)
            ptx::tc_commit_pair_mc(sfdrain_bar(sw_id), 0x1);
          else
            ptx::tc_commit(sfdrain_bar(sw_id));
          SyncCtx drain{abort_flag, p.status, p.timeout_ns};
          volatile uint32_t no_abort = 0;
          drain.abort = &no_abort;
          wait_phase(sfdrain_bar(sw_id), 0u, drain, kErrTimeoutScales);
        }
      }
      __syncwarp();
    }
  } else {
    // epilogue warpgroups: take the registers the producers gave back
    if constexpr (C::kRegSplit) ptx::setmaxnreg_inc<C::REGS_HIGH>();
    // ------------------------------------------------------------ epilogue
    if constexpr (kPair) ptx::cluster_wait();
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int epi_tid = (warp - C::EPI_WARP0) * 32 + lane;
    // the two warps of a lane quarter split the tile's columns in halves
    constexpr int kChunks = C::BN / 32;
    const int half = (warp - C::EPI_WARP0) / 4;
    const int c_begin = half * (kChunks / 2), c_end = c_begin + kChunks / 2;
    const uint32_t stg_base =
        sbase + C::OFF_STG + uint32_t((warp - C::EPI_WARP0) * C::STG_BUFS * C::STG_BYTES);
    int stg_next = 0;
    int buf = 0;
    uint32_t bphase = 0, ephase = 0;
    ptx::grid_dependency_wait();
    for (int u = group; u < units; u += ngroups) {
      const UnitCoord uc = unit_coord(u, p);
      if (!warp_wait_phase(tfull_bar(buf), bphase, sc, kErrTimeoutEpilogue)) break;
      ptx::tc_fence_after();
      const int row_in_tile = q * 32 + lane;                       // row within this CTA's 128
      const int row = uc.m_tile * C::TILE_M + int(rank) * kBM + row_in_tile;
      const int col_tile0 = uc.n_tile * C::BN;
      const int sub = uc.tile * C::CTAS + int(rank);               // split-K sub-tile index
      const bool warp_has_rows = row - lane < p.M;                 // warp-uniform
      // Convert and store 32 accumulator columns of this thread's row.
      auto store_chunk = [&](int c, const uint32_t (&r)[32]) {
        const int col0 = col_tile0 + c * 32;
        const int nvalid = min(32, p.N - col0);
        if (row >= p.M) return;
        if (p.splits > 1) {
          float* dst = p.ws + ((((size_t)sub * p.splits + uc.s) * kBM + row_in_tile) * C::BN + c * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (v * 4 < nvalid) ptx::st_global_v4(dst + v * 4, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
        } else if constexpr (C::kOutF32) {
          float* dst = reinterpret_cast<float*>(p.y) + (size_t)row * p.N + col0;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            if (v * 4 < nvalid) ptx::st_global_v4(dst + v * 4, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
        } else {
          __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.y) + (size_t)row * p.N + col0;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (v * 8 < nvalid) {
              const float* f = reinterpret_cast<const float*>(r + 8 * v);
              ptx::st_global_v4(dst + v * 8, ptx::pack_bf16x2(f[0], f[1]), ptx::pack_bf16x2(f[2], f[3]),
                                ptx::pack_bf16x2(f[4], f[5]), ptx::pack_bf16x2(f[6], f[7]));
            }
          }
        }
      };
      const uint32_t trow = tmem_base + uint32_t(buf * C::BN) + (uint32_t(q * 32) << 16);
      // Unsplit tiles: each 32 x 32 block is converted into a staging buffer (row = lane) and
      // written by one TMA store, which also clips rows >= M and columns >= N.
      auto stage_and_store = [&](int c, const uint32_t (&r)[32]) {
        const uint32_t dst = stg_base + uint32_t(stg_next * C::STG_BYTES);
        if (lane == 0) ptx::bulk_wait_read<C::STG_BUFS - 1>();   // the buffer's last store has read it
        __syncwarp();
        // The block is laid out as the TMA store's swizzle expects (16-byte chunk j of row
        // `lane` at chunk j ^ f(lane)), which also spreads a warp's stores over all banks.
        if constexpr (C::kOutF32) {
#pragma unroll
          for (int v = 0; v < 8; ++v)                   // 128-byte rows, 128-byte swizzle
            ptx::st_shared_v4(dst + lane * 128 + ((v ^ (lane & 7)) << 4), r[4 * v], r[4 * v + 1],
                              r[4 * v + 2], r[4 * v + 3]);
        } else {
#pragma unroll
          for (int v = 0; v < 4; ++v) {                 // 64-byte rows, 64-byte swizzle
            const float* f = reinterpret_cast<const float*>(r + 8 * v);
            ptx::st_shared_v4(dst + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4), ptx::pack_bf16x2(f[0], f[1]),
                              ptx::pack_bf16x2(f[2], f[3]), ptx::pack_bf16x2(f[4], f[5]),
                              ptx::pack_bf16x2(f[6], f[7]));
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&tmap_y, dst, col_tile0 + c * 32, row - lane);
          ptx::bulk_commit();
        }
        stg_next = (stg_next + 1) % C::STG_BUFS;
      };
      // The same for a block already rounded to bf16 pairs (16 words per row).
      auto stage_and_store_packed = [&](int c, const uint32_t (&pk)[16]) {
        const uint32_t dst = stg_base + uint32_t(stg_next * C::STG_BYTES);
        if (lane == 0) ptx::bulk_wait_read<C::STG_BUFS - 1>();
        __syncwarp();
#pragma unroll
        for (int v = 0; v < 4; ++v)
          ptx::st_shared_v4(dst + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4), pk[4 * v], pk[4 * v + 1],
                            pk[4 * v + 2], pk[4 * v + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&tmap_y, dst, col_tile0 + c * 32, row - lane);
          ptx::bulk_commit();
        }
        stg_next = (stg_next + 1) % C::STG_BUFS;
      };
      // Tell the MMA issuer this warp has read its part of the accumulator.
      auto release_accumulator = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) {
            ptx::fence_release_shared();
            ptx::mbar_arrive_remote_relaxed(ptx::mapa_shared(tempty_bar(buf), 0));   // the leader's
          } else {
            ptx::mbar_arrive(tempty_bar(buf));
          }
        }
      };
      constexpr int kHalfChunks = kChunks / 2;      // 32-column chunks per warp
      constexpr bool kPackedRelease = C::ACC_BUFS == 1 && C::kRegSplit && !C::kOutF32;
      if (kPackedRelease && p.splits == 1) {
        // Single accumulator (the next tile's MMAs wait for it): read all of this warp's chunks
        // out of TMEM, rounded to bf16 pairs in registers, release the accumulator, and only
        // then stage and store them while the next tile's MMAs run.
        uint32_t pk[kHalfChunks][16];
        const int nvalid =
            warp_has_rows ? max(0, min(kHalfChunks, (p.N - col_tile0 + 31) / 32 - c_begin)) : 0;
#pragma unroll
        for (int j = 0; j < kHalfChunks; ++j) {
          if (j < nvalid) {                          // uniform across the warp
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(trow + uint32_t((c_begin + j) * 32), r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 16; ++v)
              pk[j][v] = ptx::pack_bf16x2_ordered(__uint_as_float(r[2 * v]), __uint_as_float(r[2 * v + 1]));
          }
        }
        release_accumulator();
#pragma unroll
        for (int j = 0; j < kHalfChunks; ++j)
          if (j < nvalid) stage_and_store_packed(c_begin + j, pk[j]);
        if (++buf == C::ACC_BUFS) {
          buf = 0;
          bphase ^= 1u;
        }
        continue;                                  // no split-K merge on this path
      } else {
      // Two 32-column TMEM loads per wait; a warp whose 32 rows all lie past M reads nothing.
      // The accumulator is released right after this warp's last TMEM read, before that read's
      // stores: with a single accumulator the next tile's MMAs are waiting for it.
      bool released = false;
#pragma unroll 1
      for (int c = c_begin; c < c_end; c += 2) {
        if (col_tile0 + c * 32 >= p.N || !warp_has_rows) break;   // uniform across the warp
        uint32_t r0[32], r1[32];
        const bool two = c + 1 < c_end && col_tile0 + (c + 1) * 32 < p.N;
        ptx::tmem_ld_32x32b_x32(trow + uint32_t(c * 32), r0);
        if (two) ptx::tmem_ld_32x32b_x32(trow + uint32_t((c + 1) * 32), r1);
        ptx::tmem_wait_ld();
        const bool last = c + 2 >= c_end || col_tile0 + (c + 2) * 32 >= p.N;
        if (last) {
          release_accumulator();
          released = true;
        }
        if (p.splits > 1) {
          store_chunk(c, r0);
          if (two) store_chunk(c + 1, r1);
        } else if constexpr (!kPackedRelease) {      // (unsplit tiles take the path above)
          stage_and_store(c, r0);
          if (two) stage_and_store(c + 1, r1);
        }
      }
      if (!released) release_accumulator();
      }
      if (++buf == C::ACC_BUFS) {
        buf = 0;
        bphase ^= 1u;
      }
      if (p.splits > 1) {
        // Fixed-order merge of the S partials of this sub-tile: every output element sums its S
        // partials strictly in split order, ((p0 + p1) + p2) + ..., whoever computes it.  When
        // every unit has its own resident CTA group (coop_merge), the S split CTAs wait for one
        // another and each merges 1/S of the elements; otherwise the last CTA to arrive (an
        // integer counter) merges them all.
        // Hand-off 1: every partial of this CTA is stored before the count.  The barrier makes the
        // epilogue threads' stores visible to the counting thread, whose GPU-scope fence then
        // publishes them (cumulatively) before its arrival.
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(epi_bar);
        if (!warp_wait_phase(epi_bar, ephase, sc, kErrTimeoutEpilogue)) break;
        ephase ^= 1u;
        if (epi_tid == 0) {
          __threadfence();
          uint32_t* cnt = p.counters + sub;
          const uint32_t S = uint32_t(p.splits);
          bool arrive = true;
#ifdef BI_GEMM_CONTROLS
          // control build only: split 0 never counts its arrival, so the others' waits expire
          arrive = !((p.test_flags & 2u) && uc.s == 0);
#endif
          const uint32_t old = arrive ? atomicAdd(cnt, 1u) : 0u;
          uint32_t verdict = (old == S - 1) ? 1u : 0u;
          if (verdict) __threadfence();   // acquire: the other partials are visible before the merge
          if (p.coop_merge) {
            // arrivals count 0 .. S; then departures S .. 2S, and the last one out resets the
            // counter for the next launch (every CTA has seen S by then)
            const uint64_t t0 = ptx::globaltimer();
            verdict = 1u;
            for (uint32_t spin = 0; ptx::ld_acquire_gpu(cnt) < S; ++spin) {
              if ((spin & 63u) == 63u && (*abort_flag || ptx::globaltimer() - t0 > p.timeout_ns)) {
                *abort_flag = 1u;
                atomicOr(p.status, kErrTimeoutMerge);
                verdict = 0u;
                break;
              }
            }
            if (verdict && atomicAdd(cnt, 1u) == 2 * S - 1) atomicExch(cnt, 0u);
          }
          *last_flag = verdict;
        }
        // Hand-off 2: the verdict is visible to all epilogue warps.
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(epi_bar);
        if (!warp_wait_phase(epi_bar, ephase, sc, kErrTimeoutEpilogue)) break;
        ephase ^= 1u;
        const bool merge = *last_flag != 0u;
        if (merge) {
          // (row, 4-column group) items, spread over the merging CTA(s)' epilogue threads, with
          // the loads of each item issued together (see below).  The counting thread acquired
          // the partials (its fence after the last arrival, or its acquiring load of the full
          // count) before hand-off 2.
          const int row0 = uc.m_tile * C::TILE_M + int(rank) * kBM;
          const int rows = min(kBM, p.M - row0);
          const int groups = (min(C::BN, p.N - col_tile0) + 3) / 4;
          const int items = rows * groups;
          int it_begin = 0, it_end = items;
          if (p.coop_merge) {
            const int per = (items + p.splits - 1) / p.splits;
            it_begin = min(items, uc.s * per);
            it_end = min(items, it_begin + per);
          }
          const float* src0 = p.ws + ((size_t)sub * p.splits) * kBM * C::BN;
          const size_t sstride = (size_t)kBM * C::BN;
          auto store_item = [&](int rr, int g4, const float4& acc) {
            const size_t yo = (size_t)(row0 + rr) * p.N + col_tile0 + g4 * 4;
            if constexpr (C::kOutF32) {
              *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + yo) = acc;
            } else {
              uint2 pk;
              pk.x = ptx::pack_bf16x2(acc.x, acc.y);
              pk.y = ptx::pack_bf16x2(acc.z, acc.w);
              *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.y) + yo) = pk;
            }
          };
          // The epilogue's staging buffers are idle in a split run (partials go straight to
          // global memory): each merging thread copies all S partials of its item into its own
          // slot there with cp.async, so that they arrive in one round trip, then sums them.
          // Slots are padded by 16 bytes so that the threads' reads spread over the banks.
          constexpr int kStgTotal = C::EPI_WARPS * C::STG_BUFS * C::STG_BYTES;
          const int slot_bytes = p.splits * 16 + 16;
          const int per_round = min(C::EPI_THREADS, kStgTotal / slot_bytes);
          if (per_round >= 1) {
            const uint32_t slot = sbase + C::OFF_STG + uint32_t(epi_tid * slot_bytes);
#pragma unroll 1
            for (int base = it_begin; base < it_end; base += per_round) {
              const int it = base + epi_tid;
              if (epi_tid < per_round && it < it_end) {
                const int rr = it / groups, g4 = it - rr * groups;
                const float* sp = src0 + (size_t)rr * C::BN + g4 * 4;
#pragma unroll 4
                for (int s = 0; s < p.splits; ++s) ptx::cp_async_16(slot + s * 16, sp + s * sstride, 16u);
                ptx::cp_async_commit();
                ptx::cp_async_wait<0>();
                float4 acc = ptx::ld_shared_f4(slot);
#pragma unroll 4
                for (int s = 1; s < p.splits; ++s) {
                  const float4 t = ptx::ld_shared_f4(slot + s * 16);
                  acc.x = acc.x + t.x;
                  acc.y = acc.y + t.y;
                  acc.z = acc.z + t.z;
                  acc.w = acc.w + t.w;
                }
                store_item(rr, g4, acc);
              }
            }
          } else {
            // S too large for the staging: loads in registers, in batches
#pragma unroll 1
            for (int it = it_begin + epi_tid; it < it_end; it += C::EPI_THREADS) {
              const int rr = it / groups, g4 = it - rr * groups;
              const float* sp = src0 + (size_t)rr * C::BN + g4 * 4;
              constexpr int kMergeBatch = C::kRegSplit ? 4 : 16;   // loads in flight per item
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
              for (int s0 = 0; s0 < p.splits; s0 += kMergeBatch) {
                float4 t[kMergeBatch];
#pragma unroll
                for (int j = 0; j < kMergeBatch; ++j)
                  if (s0 + j < p.splits) t[j] = __ldcg(reinterpret_cast<const float4*>(sp + (s0 + j) * sstride));
                int j0 = 0;
                if (s0 == 0) {                   // the sum starts from p0 itself, not 0 + p0
                  acc = t[0];
                  j0 = 1;
                }
#pragma unroll
                for (int j = 0; j < kMergeBatch; ++j) {
                  if (j >= j0 && s0 + j < p.splits) {
                    acc.x = acc.x + t[j].x;
                    acc.y = acc.y + t[j].y;
                    acc.z = acc.z + t[j].z;
                    acc.w = acc.w + t[j].w;
                  }
                }
              }
              store_item(rr, g4, acc);
            }
          }
          if (!p.coop_merge && epi_tid == 0) p.counters[sub] = 0u;   // ready for the next launch
        }
        // Hand-off 3: last_flag may be rewritten only after every warp has read it.
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(epi_bar);
        if (!warp_wait_phase(epi_bar, ephase, sc, kErrTimeoutEpilogue)) break;
        ephase ^= 1u;
      }
    }
  }

  // the output stores must have read their staging buffers before shared memory is released
  if (warp >= C::EPI_WARP0 && lane == 0) ptx::bulk_wait_read<0>();
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (kPair) ptx::cluster_sync();   // neither CTA leaves while the pair still works
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (kPair)
      ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace bigemm
