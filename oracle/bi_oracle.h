/*
 * bi_oracle.h — plain, slow CPU oracle for the batch-invariant GEMM y = x·W
 * (and the batch-invariant RMSNorm, decode attention and mHC pre-norm projection, declared at
 * the end).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The product path (the CUDA library and
 * its Python binding) never calls it and shares no code with it.
 *
 * What it computes (the plain definition, "Batch-invariant matrix multiplication",
 * nondeterminism article: C_ij = sum_k A_ik B_kj, with the whole K reduction of one
 * output kept in one place):
 *
 *     acc[i,j]  = sum_{k=0..K-1, ascending} dec(x[i,k]) * dec(w[k,j])     (fp64)
 *     sabs[i,j] = sum_{k=0..K-1, ascending} |dec(x[i,k]) * dec(w[k,j])|   (fp64)
 *     y[i,j]    = round_out(acc[i,j])      one round-to-nearest-even, fp64 -> out
 *
 * Layouts: x[M,K] row-major, w[K,N] row-major, y[M,N] row-major.  Each output row
 * is computed from its own input row only (the definition y[i] = f(x[i], W) of the
 * batch-invariance issue, "Problem statement").
 *
 * Decoding (all exact in fp64):
 *   bf16:   bit pattern << 16 is the fp32 pattern of the same value.
 *   E4M3FN: sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0 = subnormal
 *           m * 2^-9; S.1111.111 = NaN; no infinities; max 448.
 *   E8M0:   value 2^(e - 127); 0xFF = NaN.
 *   MXFP8 element: e4m3(x[i,k]) * 2^(sx[i, k/32] - 127), e4m3(w[k,j]) * 2^(sw[k/32, j] - 127).
 *
 * Products of two decoded bf16 (8-bit significands) or two decoded E4M3 values are
 * exact in fp64; the fp64 running sum rounds only when its magnitude range exceeds
 * 53 bits.  Output rounding is a single RNE step from fp64 straight to the output type.
 *
 * Errors: functions return 0 on success, -1 on a bad argument (null pointer with a
 * non-zero size, negative size).  No allocation escapes a call.
 */
#ifndef BI_ORACLE_H
#define BI_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { BIO_OUT_BF16 = 0, BIO_OUT_F32 = 1 };

/* Scalar decoders / encoders (exposed so the tests can pin them on their own). */
double   bio_bf16_to_f64(uint16_t b);
double   bio_e4m3_to_f64(uint8_t c);
double   bio_e8m0_to_f64(uint8_t e);
uint16_t bio_f64_to_bf16(double v);   /* single RNE rounding, overflow -> inf */
uint32_t bio_f64_to_f32(double v);    /* single RNE rounding, returns the bit pattern */

/* Core: fp64 inputs, fp64 outputs (no output rounding).  acc/sabs are [M,N]; sabs may be NULL. */
int bio_gemm_f64(const double* x, int64_t M, int64_t K, const double* w, int64_t N,
                 double* acc, double* sabs);

/* bf16 inputs.  rows: optional list of nrows row indices of x to compute (NULL = all M rows,
 * nrows ignored); outputs are packed [nrows or M, N].  y: uint16 bf16 patterns (out=BF16) or
 * uint32 fp32 patterns (out=F32).  acc and sabs (fp64, same packing) may be NULL. */
int bio_gemm_bf16(const uint16_t* x, int64_t M, int64_t K, const uint16_t* w, int64_t N,
                  const int64_t* rows, int64_t nrows, int out, void* y, double* acc, double* sabs);

/* MXFP8 inputs: x E4M3 [M,K], sx E8M0 [M,K/32], w E4M3 [K,N], sw E8M0 [K/32,N]; K % 32 == 0.
 * Output bf16 (uint16 patterns) [nrows or M, N]; rows/acc/sabs as for bio_gemm_bf16. */
int bio_gemm_mxfp8(const uint8_t* x, const uint8_t* sx, int64_t M, int64_t K,
                   const uint8_t* w, const uint8_t* sw, int64_t N,
                   const int64_t* rows, int64_t nrows, uint16_t* y, double* acc, double* sabs);

/* RMSNorm of bf16 rows ("Batch-invariant RMSNorm", nondeterminism article: RMSNorm(x_i) =
 * x_i / sqrt(mean_j x_ij^2 + eps) * gamma, one reduction along the feature axis per row):
 *
 *     ms[i]   = (sum_{j=0..d-1, ascending} x[i,j]^2) / d          (fp64)
 *     r[i]    = 1 / sqrt(ms[i] + eps)                              (fp64)
 *     v[i,j]  = (x[i,j] * r[i]) * g[j]                             (fp64, the article's order
 *                                                                   x * rsqrt(mean) * weight)
 *     y[i,j]  = RNE bf16 of v[i,j]
 *
 * x[M,d] and y bf16 patterns row-major, g[d] bf16 patterns.  rows/nrows select rows as for
 * bio_gemm_bf16.  v (fp64, same packing as y) may be NULL; it is the unrounded value the
 * tolerance is measured against.  Returns -1 on a bad argument (negative sizes, d = 0 with
 * M > 0, NaN or negative eps). */
int bio_rmsnorm_bf16(const uint16_t* x, int64_t M, int64_t d, const uint16_t* g, double eps,
                     const int64_t* rows, int64_t nrows, uint16_t* y, double* v);

/* Causal attention of query tokens over a paged bf16 KV cache ("Batch-invariant attention",
 * nondeterminism article: O_i = sum_{j <= i} softmax(q_i . k_j / sqrt(d)) v_j, with the K/V
 * cache filled before the attention runs).  For query token t (request b = q_seq[t], position
 * p = q_pos[t]) and query head h (KV head h / G, G = Hq / Hkv):
 *
 *     s_j   = scale * sum_{i ascending} q[t,h,i] * K_b[j, h/G, i]          j = 0..p  (fp64)
 *     m     = max_j s_j,   w_j = exp(s_j - m)
 *     v[i]  = (sum_{j ascending} w_j * V_b[j, h/G, i]) / (sum_{j ascending} w_j)
 *     o     = RNE bf16 of v
 *
 * K_b[j, kh, i] = k_cache[page_table[b * max_pages + j / page_size], j % page_size, kh, i]
 * (V alike); k_cache and v_cache are [num_pages, page_size, Hkv, D] bf16 patterns, q and o
 * [T, Hq, D].  Optional fp64 outputs, [T, Hq, D] unless noted: v (unrounded), a = (sum_j w_j
 * |V_b[j, h/G, i]|) / (sum_j w_j) and, per [T, Hq], e = max_j scale * sum_i |q_i K_b[j, i]|
 * (the scale of the score rounding errors) — both for the tolerance.  Returns -1 on a bad
 * argument (sizes, Hq % Hkv, a position or page index out of range). */
int bio_attention_bf16(const uint16_t* q, int64_t T, int64_t Hq, int64_t D,
                       const int32_t* q_seq, const int32_t* q_pos,
                       const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_pages,
                       int64_t page_size, int64_t Hkv, const int32_t* page_table, int64_t B,
                       int64_t max_pages, double scale, uint16_t* o, double* v, double* a, double* e);

/* Pre-norm projection of the hyper-connection ("mHC") block ("[BI][DSv4] Make mHC tilelang ops
 * batch invariant": the prenorm GEMM that projects the flattened streams, with its fused
 * RMSNorm): for each row i of x[M,K] (bf16 patterns) and W[K,N] (bf16 patterns), in fp64,
 *
 *     a[i,j] = sum_{k ascending} x[i,k] * W[k,j]
 *     ss[i]  = sum_{k ascending} x[i,k]^2
 *     v[i,j] = a[i,j] / sqrt(ss[i] / K + eps)        (RMSNorm(x_i) . W, no norm weight)
 *     y[i,j] = RNE fp32 of v[i,j]                     (uint32 patterns)
 *
 * Optional fp64 outputs: v (unrounded) and sabs[i,j] = (sum_k |x W|) / sqrt(ss/K + eps), the
 * scale of the rounding errors.  Returns -1 on a bad argument (sizes, NaN or negative eps). */
int bio_prenorm_gemm(const uint16_t* x, int64_t M, int64_t K, const uint16_t* w, int64_t N, double eps,
                     uint32_t* y, double* v, double* sabs);

#ifdef __cplusplus
}
#endif
#endif
