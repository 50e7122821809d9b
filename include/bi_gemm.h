/*
 * bi_gemm.h — C ABI of the batch-invariant GEMM library (libbi_gemm.so), sm_103a (GB300).
 *
 *     y[M, N] = x[M, K] · W[K, N]        fp32 accumulation
 *
 * Batch invariance is the row-wise definition y[i] = f(x[i], W) of the batch-invariance
 * test issue (gitcode.com/CANN/ops-transformer/issues/2956, "Problem statement"): output
 * row i depends only on input row i and the shared W, bit for bit, for every M and every
 * content of the other rows.  The library gets it the way the nondeterminism article
 * prescribes ("Batch-invariant matrix multiplication": compile one kernel configuration
 * and use it for every shape): the tile shape, tcgen05 instruction shape, K order and
 * split count are chosen once at bi_gemm_create from (K, N, dtype, scale_layout, SM
 * count) and never from M.  Where a split count S > 1 is chosen, split s always covers
 * the same K range and the S partials are merged in one fixed serial order ("[BI][DSv4]
 * Make mHC tilelang ops batch invariant", "What": a pinned split count with a serial
 * merge pins the reduction tree).  Results are also identical from run to run (no
 * floating-point atomics; nondeterminism article, "Three kinds of determinism").
 * Bit equality with other GPUs, drivers or library versions is not claimed.
 *
 * Conventions shared by all entry points:
 *   - Return value: BI_GEMM_OK (0) or a negative BI_GEMM_ERR_* code; no entry point aborts
 *     the process or prints.  bi_gemm_strerror() names a code.
 *   - Layouts: row-major.  x is [M, K] (K contiguous), W is [K, N] (N contiguous), y is
 *     [M, N] (N contiguous); no strides or transposes.
 *   - Data pointers are DEVICE pointers owned by the caller, on the device that was
 *     current at bi_gemm_create; they must stay valid until the work queued on `stream`
 *     has finished.  `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - A handle is not thread-safe and must not be used on two streams at once.
 *   - There is no fallback: a shape or layout the fixed configuration cannot serve is
 *     refused at bi_gemm_create (fail closed), never routed to another kernel.
 */
#ifndef BI_GEMM_H
#define BI_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bi_gemm* bi_gemm_t;

/* Input and output element types. */
typedef enum {
  BI_BF16_OUT_BF16 = 0,       /* x, W bf16; y bf16 (round to nearest even from fp32)     */
  BI_BF16_OUT_F32 = 1,        /* x, W bf16; y fp32                                        */
  BI_MXFP8E4M3_OUT_BF16 = 2   /* x, W OCP E4M3FN with E8M0 block scales; y bf16          */
} bi_gemm_dtype;

/* Scale layout.  BI_SCALES_E8M0_K32 (MXFP8 only): one E8M0 exponent per 32 consecutive K
 * elements — sx[M, K/32] for the rows of x and sw[K/32, N] for the columns of W, both
 * row-major uint8 (value 2^(e-127)); block kb covers k in [32*kb, 32*kb + 32).  This is the
 * block-scaled MXFP8 format whose K-axis-varying scales are the known batch-invariance
 * trigger of the batch-invariance test issue ("Test methodology"). */
typedef enum {
  BI_SCALES_NONE = 0,
  BI_SCALES_E8M0_K32 = 1
} bi_gemm_scale_layout;

/* Device pointers to the two scale matrices (MXFP8 only). */
typedef struct {
  const uint8_t* sx; /* [M, K/32] E8M0, 4-byte aligned (else BI_GEMM_ERR_ALIGNMENT) */
  const uint8_t* sw; /* [K/32, N] E8M0, 16-byte aligned (else BI_GEMM_ERR_ALIGNMENT) */
} bi_gemm_scales;

enum {
  BI_GEMM_OK = 0,
  BI_GEMM_ERR_INVALID_ARG = -1,  /* null handle / pointer, negative size, bad enum        */
  BI_GEMM_ERR_UNSUPPORTED = -2,  /* shape or dtype the fixed configuration cannot serve    */
  BI_GEMM_ERR_ALIGNMENT = -3,    /* a pointer or row pitch breaks the 16-byte rule          */
  BI_GEMM_ERR_CUDA = -4,         /* a CUDA runtime call failed (launch, allocation setup)   */
  BI_GEMM_ERR_OOM = -5,          /* workspace allocation failed                             */
  BI_GEMM_ERR_TIMEOUT = -6,      /* a bounded in-kernel wait expired (reported by
                                    bi_gemm_get_device_error)                               */
  BI_GEMM_ERR_SCRATCH_LIMIT = -7 /* bi_gemm_run_noalloc: the run needs more scratch than its
                                    fixed array holds                                       */
};

/* Create a handle for y = x·W with fixed K and N.  Selects and records the single kernel
 * configuration (tile, instruction shape, pipeline depth, split count) from K, N, dtype,
 * scale_layout and the current device's SM count; M is not an input.  Allocates a 4-byte
 * device status word.  Requirements (else BI_GEMM_ERR_UNSUPPORTED): K >= 1, N >= 1,
 * K, N < 2^31; bf16: K % 8 == 0 and N % 8 == 0 (16-byte row pitch); MXFP8: K % 128 == 0
 * and N % 16 == 0, scale_layout == BI_SCALES_E8M0_K32; bf16: scale_layout == BI_SCALES_NONE.
 * The device must be compute capability 10.3 (sm_103a).  On success *out owns the handle;
 * release it with bi_gemm_destroy. */
int bi_gemm_create(bi_gemm_t* out, int64_t K, int64_t N, int dtype, int scale_layout);

/* Options for bi_gemm_create_ex.  Zero-initialise, then set what you need. */
typedef struct {
  int32_t split_k;        /* 0 = automatic (the rule above); >= 1 forces this fixed split
                             count (1 <= split_k <= ceil(K / BK)); still never M-dependent */
  int32_t max_ctas;       /* 0 = one CTA per SM; otherwise an upper bound on the grid     */
  uint64_t timeout_ns;    /* 0 = default (5 s); limit of every in-kernel wait             */
  uint32_t flags;         /* OR of BI_GEMM_FLAG_* below; 0 = none                          */
  uint32_t reserved;      /* must be 0                                                     */
} bi_gemm_options;

/* BI_GEMM_FLAG_STATIC_W: the caller guarantees that no kernel which may still be running when
 * a run is queued writes that run's W (typical for inference weights).  Each run then starts
 * loading its first W tiles while the previous kernel in the stream is still finishing, and
 * only the x loads wait for that kernel (programmatic dependent launch); this hides part of
 * the launch latency of back-to-back runs.  It changes no arithmetic and no result.  Without
 * the flag every global load of a run waits for the previous kernel to complete. */
#define BI_GEMM_FLAG_STATIC_W 1u

/* bi_gemm_create with explicit options (NULL = defaults, same as bi_gemm_create). */
int bi_gemm_create_ex(bi_gemm_t* out, int64_t K, int64_t N, int dtype, int scale_layout,
                      const bi_gemm_options* opt);

/* Enqueue y = x·W on `stream`.  M >= 0 rows (M == 0 is a no-op that returns BI_GEMM_OK).
 * x, W, y: device pointers, 16-byte aligned.  scales: NULL for bf16; for MXFP8 a host
 * struct holding the two device scale pointers.  Asynchronous: returns after queuing.
 * When the handle's split count is > 1 the handle grows its workspace (fp32 partials,
 * tiles*S*128*BN*4 bytes, plus one arrival counter per tile) with stream-ordered
 * allocation on `stream` the first time a larger M needs it; BI_GEMM_ERR_OOM if that fails.
 * Errors from the kernel's bounded waits are reported by bi_gemm_get_device_error. */
int bi_gemm_run(bi_gemm_t h, const void* x, int64_t M, const void* W,
                const bi_gemm_scales* scales, void* y, void* stream);

/* One row block of a gathered run: x [rows, K] (device pointer, 16-byte aligned, rows contiguous)
 * and, for MXFP8, its scales sx [rows, K/32] (device pointer, 4-byte aligned; NULL for bf16). */
typedef struct {
  const void* x;
  const uint8_t* sx;
  int64_t rows;
} bi_gemm_block;

/* Gather + GEMM: the all-gather matmul of the batch-invariance test issue ("Background": each
 * rank's row block of x is gathered, then multiplied by the shared W, and the defect was one
 * kernel for the local rows and another for the gathered ones).  The nblocks blocks, in order
 * (say rank 0's, rank 1's, ...; all in this GPU's memory: in a multi-rank run the caller's
 * collective has delivered them), are copied into x_out [M, K], M = the sum of their rows (and,
 * for MXFP8, their scales into sx_out [M, K/32]); then y [M, N] = x_out · W runs on the handle
 * exactly as bi_gemm_run, with its one kernel configuration for every row.  So a row's output bits
 * do not depend on which block it came from or on the other blocks, and equal those of
 * bi_gemm_run on its block alone.  sw: W's scales [K/32, N] for MXFP8 (16-byte aligned), NULL for
 * bf16.  1 <= nblocks <= 256; a block may have 0 rows.  x_out (16-byte aligned) and sx_out
 * (4-byte aligned) are caller-owned and must not overlap the blocks.  Asynchronous on `stream`;
 * errors as bi_gemm_run, and BI_GEMM_ERR_INVALID_ARG for a bad block table. */
int bi_gemm_run_gathered(bi_gemm_t h, const bi_gemm_block* blocks, int32_t nblocks, void* x_out,
                         uint8_t* sx_out, const void* W, const uint8_t* sw, void* y, void* stream);

/* Allocation-free variant of bi_gemm_run (the papers have no counterpart; this is a service
 * of this library).  It is for callers that may not allocate device memory when they run a
 * GEMM: code whose device memory is wholly owned and budgeted by another framework's pool,
 * latency-critical loops that must not enter the allocator (its locks and implicit
 * synchronisation), and code running where CUDA allocation calls are not permitted.
 * Same arguments, layouts, kernel and results as bi_gemm_run on the same handle; the
 * difference is where a split count S > 1 keeps its scratch (one uint32 arrival counter per
 * output tile and tiles*S*128*BN fp32 partials): instead of the handle's workspace, grown with
 * cudaMallocAsync, it uses one fixed 8 MiB device array compiled into the library (4 KiB of
 * counters, then 8 MiB - 4 KiB of partials).  Every GPU on which
 * the library's kernels are loaded holds that array until the process exits.  This call makes
 * no cudaMalloc, cudaMallocAsync or cudaFree and calls no allocating library routine.
 *   - The first call in each CUDA context looks up the array's device address there
 *     (cudaGetSymbolAddress, with the handle's device current) and keeps it with the
 *     context's unique id; later calls in that context reuse it, and a context created later
 *     (for instance after cudaDeviceReset, which reloads the module) gets a fresh lookup.
 *     Make that first call before any stream capture.  The handle's device must be current
 *     (else BI_GEMM_ERR_INVALID_ARG).
 *   - A run whose scratch would not fit returns BI_GEMM_ERR_SCRATCH_LIMIT and queues nothing:
 *     tiles*S*128*BN*4 bytes of partials must be <= 8 MiB - 4 KiB, where tiles, the 128-row
 *     sub-tiles, is ceil(M/block_m) * ctas_per_tile * ceil(N/BN) (bi_gemm_get_config gives
 *     block_m, ctas_per_tile, S and BN).  This is the bound that binds: it admits at most 127
 *     sub-tiles, and the 4 KiB of counters hold 1024.  Handles with S == 1 use no scratch.
 *   - All calls in the process share the one array per device and it keeps the last call's
 *     contents; each call first clears, on `stream`, the counters it uses.  Calls whose work
 *     overlaps on the GPU (other streams, other threads, other handles) race on the array and
 *     give undefined results: serialise them. */
int bi_gemm_run_noalloc(bi_gemm_t h, const void* x, int64_t M, const void* W,
                        const bi_gemm_scales* scales, void* y, void* stream);

/* Synchronise `stream`, then read and clear the handle's device status word: BI_GEMM_OK,
 * or BI_GEMM_ERR_TIMEOUT if any run since the last call had a bounded wait expire (its
 * output is then undefined), or BI_GEMM_ERR_CUDA if synchronisation failed. */
int bi_gemm_get_device_error(bi_gemm_t h, void* stream);

/* Release the handle, its status word and its workspace (synchronises the device first).
 * NULL is accepted. */
int bi_gemm_destroy(bi_gemm_t h);

/* The fixed configuration recorded in a handle. */
typedef struct {
  int32_t block_m, block_n, block_k;  /* output tile rows / columns, K per pipeline stage
                                         (a CTA pair's tile is 256 x 256)                   */
  int32_t mma_m, mma_n, mma_k;        /* tcgen05.mma instruction shape                     */
  int32_t stages;                     /* shared-memory pipeline depth                       */
  int32_t split_k;                    /* S: fixed K split count (1 = none)                  */
  int32_t num_sms;                    /* SMs on the device at create                        */
  int32_t max_ctas;                   /* grid upper bound                                   */
  int32_t threads;                    /* threads per CTA                                    */
  int32_t smem_bytes;                 /* dynamic shared memory per CTA                      */
  int32_t tmem_cols;                  /* tensor-memory columns per CTA                      */
  int32_t ctas_per_tile;              /* 1, or 2 for a CTA-pair tile (tcgen05 cta_group::2) */
  int32_t max_groups;                 /* resident CTA groups (CTAs or pairs) in the grid    */
} bi_gemm_config;

int bi_gemm_get_config(bi_gemm_t h, bi_gemm_config* cfg);

/* Bytes of workspace a run with M rows needs on this handle (0 when split_k == 1). */
int bi_gemm_workspace_size(bi_gemm_t h, int64_t M, uint64_t* bytes);

/* Static description of an error code (never NULL). */
const char* bi_gemm_strerror(int code);

/* Library ABI version: (major << 16) | minor. */
int bi_gemm_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BI_GEMM_H */
