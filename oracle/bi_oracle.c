/*
 * bi_oracle.c — plain CPU oracle for the batch-invariant GEMM, RMSNorm and attention (TEST
 * INFRASTRUCTURE).
 *
 * Only tests, the smoke check and the benchmark's CPU-baseline leg use this file.
 * It follows the plain definition C_ij = sum_k A_ik B_kj of the nondeterminism
 * article ("Batch-invariant matrix multiplication"), one output row from one input
 * row (batch-invariance issue, "Problem statement": y[i] = f(x[i], W)), summing in
 * ascending k in fp64 and rounding once to the output type.
 *
 * Loop order: for each row i, for each k, for each column j, acc[j] += a_ik * w_kj.
 * Every output element still receives its K products in ascending k, one at a time,
 * exactly as the (i, j, k) order would give them; only independent elements are
 * interleaved, so no sum is reordered, blocked or fused.  Build with
 * -ffp-contract=off so that a product and the following add are never fused.
 */
#include "bi_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ decoders */

double bio_bf16_to_f64(uint16_t b) {
    /* bf16 is the upper half of an fp32 pattern. */
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double bio_e4m3_to_f64(uint8_t c) {
    int sign = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;          /* S.1111.111 */
    if (e == 0) v = ldexp((double)m, -9);           /* subnormal: m/8 * 2^(1-7) */
    else v = ldexp(8.0 + m, e - 7 - 3);             /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

double bio_e8m0_to_f64(uint8_t e) {
    if (e == 0xFF) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* --------------------------------------------------------------- encoders */

uint32_t bio_f64_to_f32(double v) {
    /* C conversion double -> float rounds to nearest, ties to even, in one step. */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

uint16_t bio_f64_to_bf16(double v) {
    uint64_t u;
    memcpy(&u, &v, sizeof u);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    int64_t e = (int64_t)((u >> 52) & 0x7FF);
    uint64_t frac = u & 0x000FFFFFFFFFFFFFull;
    if (e == 0x7FF) return frac ? (uint16_t)(sign | 0x7FC0u) : (uint16_t)(sign | 0x7F80u);
    if (e == 0 && frac == 0) return sign;
    /* |v| = sig * 2^(exp2) with sig a 53-bit integer (or smaller for fp64 subnormals). */
    uint64_t sig;
    int64_t exp2;
    if (e == 0) { sig = frac; exp2 = -1074; }
    else { sig = frac | (1ull << 52); exp2 = e - 1075; }
    /* bf16 normal: (128 + m) * 2^(E - 134) with E in [1, 254]; subnormal: m * 2^-133.
     * Find the quantum q = 2^qe of the bf16 binade that holds |v|. */
    int top = 63 - __builtin_clzll(sig);            /* |v| in [2^(top+exp2), 2^(top+exp2+1)) */
    int64_t lg = top + exp2;                        /* floor(log2 |v|) */
    int64_t qe = (lg < -126 ? -126 : lg) - 7;       /* bf16 quantum exponent */
    /* q_units = |v| / 2^qe rounded to nearest even.  shift = qe - exp2 >= 0 drops bits. */
    int64_t shift = qe - exp2;
    uint64_t units;
    if (shift <= 0) {
        units = sig << (-shift);                    /* exact (only for huge/small exps, unreachable in practice) */
    } else if (shift >= 64) {
        units = 0;                                  /* below half the smallest quantum */
        if (shift == 64 && sig > (1ull << 63)) units = 1;
    } else {
        uint64_t kept = sig >> shift;
        uint64_t rem = sig & ((1ull << shift) - 1);
        uint64_t half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (kept & 1))) kept += 1;
        units = kept;
    }
    /* value = units * 2^qe.  Encode: normal range has units in [128, 256). */
    if (qe == -133) {
        /* Subnormals (units < 128), the first normal binade (E = 1, units in [128, 256))
         * and its carry (units = 256 -> E = 2, m = 0) share the quantum 2^-133, and the
         * bf16 pattern of units * 2^-133 is the integer units itself in all three cases. */
        return (uint16_t)(sign | (uint16_t)units);
    }
    if (units == 256) { units = 128; qe += 1; }     /* carry into the next binade */
    int64_t E = qe + 134;                           /* biased exponent */
    if (E >= 255) return (uint16_t)(sign | 0x7F80u);/* overflow -> infinity */
    return (uint16_t)(sign | (uint16_t)(E << 7) | (uint16_t)(units - 128));
}

/* ------------------------------------------------------------------ GEMMs */

int bio_gemm_f64(const double* x, int64_t M, int64_t K, const double* w, int64_t N,
                 double* acc, double* sabs) {
    if (M < 0 || K < 0 || N < 0) return -1;
    if ((M * N > 0) && !acc) return -1;
    if ((M * K > 0 && !x) || (K * N > 0 && !w)) return -1;
    for (int64_t i = 0; i < M; ++i) {
        double* a = acc + i * N;
        double* s = sabs ? sabs + i * N : NULL;
        for (int64_t j = 0; j < N; ++j) { a[j] = 0.0; if (s) s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double xv = x[i * K + k];
            const double* wr = w + k * N;
            for (int64_t j = 0; j < N; ++j) {
                double p = xv * wr[j];
                a[j] = a[j] + p;
                if (s) s[j] = s[j] + fabs(p);
            }
        }
    }
    return 0;
}

static void store_out(int out, void* y, int64_t idx, double v) {
    if (out == BIO_OUT_BF16) ((uint16_t*)y)[idx] = bio_f64_to_bf16(v);
    else ((uint32_t*)y)[idx] = bio_f64_to_f32(v);
}

int bio_gemm_bf16(const uint16_t* x, int64_t M, int64_t K, const uint16_t* w, int64_t N,
                  const int64_t* rows, int64_t nrows, int out, void* y, double* acc, double* sabs) {
    if (M < 0 || K < 0 || N < 0 || (out != BIO_OUT_BF16 && out != BIO_OUT_F32)) return -1;
    int64_t R = rows ? nrows : M;
    if (R < 0) return -1;
    if (R > 0 && N > 0 && !y) return -1;
    if ((M * K > 0 && !x) || (K * N > 0 && !w)) return -1;
    double* a = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!a || !s) { free(a); free(s); return -1; }
    for (int64_t r = 0; r < R; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) { free(a); free(s); return -1; }
        for (int64_t j = 0; j < N; ++j) { a[j] = 0.0; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double xv = bio_bf16_to_f64(x[i * K + k]);
            const uint16_t* wr = w + k * N;
            for (int64_t j = 0; j < N; ++j) {
                double p = xv * bio_bf16_to_f64(wr[j]);
                a[j] = a[j] + p;
                s[j] = s[j] + fabs(p);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            store_out(out, y, r * N + j, a[j]);
            if (acc) acc[r * N + j] = a[j];
            if (sabs) sabs[r * N + j] = s[j];
        }
    }
    free(a);
    free(s);
    return 0;
}

int bio_gemm_mxfp8(const uint8_t* x, const uint8_t* sx, int64_t M, int64_t K,
                   const uint8_t* w, const uint8_t* sw, int64_t N,
                   const int64_t* rows, int64_t nrows, uint16_t* y, double* acc, double* sabs) {
    if (M < 0 || K < 0 || N < 0 || (K % 32) != 0) return -1;
    int64_t R = rows ? nrows : M;
    if (R < 0) return -1;
    if (R > 0 && N > 0 && !y) return -1;
    if ((M * K > 0 && (!x || !sx)) || (K * N > 0 && (!w || !sw))) return -1;
    const int64_t KB = K / 32;
    double* a = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!a || !s) { free(a); free(s); return -1; }
    for (int64_t r = 0; r < R; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) { free(a); free(s); return -1; }
        for (int64_t j = 0; j < N; ++j) { a[j] = 0.0; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double xv = bio_e4m3_to_f64(x[i * K + k]) * bio_e8m0_to_f64(sx[i * KB + k / 32]);
            const uint8_t* wr = w + k * N;
            const uint8_t* swr = sw + (k / 32) * N;
            for (int64_t j = 0; j < N; ++j) {
                double wv = bio_e4m3_to_f64(wr[j]) * bio_e8m0_to_f64(swr[j]);
                double p = xv * wv;
                a[j] = a[j] + p;
                s[j] = s[j] + fabs(p);
            }
        }
        for (int64_t j = 0; j < N; ++j) {
            y[r * N + j] = bio_f64_to_bf16(a[j]);
            if (acc) acc[r * N + j] = a[j];
            if (sabs) sabs[r * N + j] = s[j];
        }
    }
    free(a);
    free(s);
    return 0;
}

/* ---------------------------------------------------------------- RMSNorm */

/* One row at a time, straight from the definition ("Batch-invariant RMSNorm", nondeterminism
 * article): the sum of squares in ascending j, the mean, the reciprocal square root, then
 * each element times it and times its weight, all in fp64, with one rounding to bf16. */
int bio_rmsnorm_bf16(const uint16_t* x, int64_t M, int64_t d, const uint16_t* g, double eps,
                     const int64_t* rows, int64_t nrows, uint16_t* y, double* v) {
    if (M < 0 || d < 0 || !(eps >= 0.0)) return -1;
    int64_t R = rows ? nrows : M;
    if (R < 0) return -1;
    if (R > 0 && d == 0) return -1;
    if (R > 0 && (!x || !g || !y)) return -1;
    for (int64_t r = 0; r < R; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) return -1;
        const uint16_t* xr = x + i * d;
        double ss = 0.0;
        for (int64_t j = 0; j < d; ++j) {
            const double xv = bio_bf16_to_f64(xr[j]);
            ss = ss + xv * xv;
        }
        const double ms = ss / (double)d;
        const double rr = 1.0 / sqrt(ms + eps);
        for (int64_t j = 0; j < d; ++j) {
            const double val = (bio_bf16_to_f64(xr[j]) * rr) * bio_bf16_to_f64(g[j]);
            y[r * d + j] = bio_f64_to_bf16(val);
            if (v) v[r * d + j] = val;
        }
    }
    return 0;
}

/* -------------------------------------------------------------- attention */

/* Straight from the definition ("Batch-invariant attention", nondeterminism article): for each
 * query token and head, the scores of the keys at positions 0..p, their maximum, the weights
 * exp(s - max), and the weighted mean of the values, all in fp64, rounded once to bf16. */
int bio_attention_bf16(const uint16_t* q, int64_t T, int64_t Hq, int64_t D,
                       const int32_t* q_seq, const int32_t* q_pos,
                       const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_pages,
                       int64_t page_size, int64_t Hkv, const int32_t* page_table, int64_t B,
                       int64_t max_pages, double scale, uint16_t* o, double* v, double* a, double* e) {
    if (T < 0 || Hq <= 0 || D <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_pages < 0 || page_size <= 0 ||
        B < 0 || max_pages < 0)
        return -1;
    if (T == 0) return 0;
    if (!q || !q_seq || !q_pos || !k_cache || !v_cache || !page_table || !o) return -1;
    const int64_t G = Hq / Hkv;
    /* validate every position and page first */
    for (int64_t t = 0; t < T; ++t) {
        const int64_t b = q_seq[t], p = q_pos[t];
        if (b < 0 || b >= B || p < 0 || p / page_size >= max_pages) return -1;
        for (int64_t pg = 0; pg <= p / page_size; ++pg) {
            const int64_t page = page_table[b * max_pages + pg];
            if (page < 0 || page >= num_pages) return -1;
        }
    }
    double* w = NULL;
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    double* aab = (double*)malloc(sizeof(double) * (size_t)D);
    if (!acc || !aab) { free(acc); free(aab); return -1; }
    for (int64_t t = 0; t < T; ++t) {
        const int64_t b = q_seq[t], p = q_pos[t];
        double* ww = (double*)realloc(w, sizeof(double) * (size_t)(p + 1));
        if (!ww) { free(w); free(acc); free(aab); return -1; }
        w = ww;
        for (int64_t h = 0; h < Hq; ++h) {
            const int64_t kh = h / G;
            const uint16_t* qv = q + (t * Hq + h) * D;
            double m = -INFINITY, emax = 0.0;
            for (int64_t j = 0; j <= p; ++j) {
                const int64_t page = page_table[b * max_pages + j / page_size];
                const uint16_t* kr = k_cache + ((page * page_size + j % page_size) * Hkv + kh) * D;
                double sdot = 0.0, sabs = 0.0;
                for (int64_t i = 0; i < D; ++i) {
                    const double prod = bio_bf16_to_f64(qv[i]) * bio_bf16_to_f64(kr[i]);
                    sdot = sdot + prod;
                    sabs = sabs + fabs(prod);
                }
                w[j] = scale * sdot;
                if (w[j] > m) m = w[j];
                if (scale * sabs > emax) emax = scale * sabs;
            }
            double l = 0.0;
            for (int64_t j = 0; j <= p; ++j) {
                w[j] = exp(w[j] - m);
                l = l + w[j];
            }
            for (int64_t i = 0; i < D; ++i) { acc[i] = 0.0; aab[i] = 0.0; }
            for (int64_t j = 0; j <= p; ++j) {
                const int64_t page = page_table[b * max_pages + j / page_size];
                const uint16_t* vr = v_cache + ((page * page_size + j % page_size) * Hkv + kh) * D;
                for (int64_t i = 0; i < D; ++i) {
                    const double vv = bio_bf16_to_f64(vr[i]);
                    acc[i] = acc[i] + w[j] * vv;
                    aab[i] = aab[i] + w[j] * fabs(vv);
                }
            }
            const int64_t base = (t * Hq + h) * D;
            for (int64_t i = 0; i < D; ++i) {
                const double val = acc[i] / l;
                o[base + i] = bio_f64_to_bf16(val);
                if (v) v[base + i] = val;
                if (a) a[base + i] = aab[i] / l;
            }
            if (e) e[t * Hq + h] = emax;
        }
    }
    free(w);
    free(acc);
    free(aab);
    return 0;
}

/* ---------------------------------------------------------- mHC pre-norm GEMM */

/* One row at a time, from the definition: the projection and the sum of squares in ascending k
 * (fp64), then the projection divided by the root mean square, rounded once to fp32. */
int bio_prenorm_gemm(const uint16_t* x, int64_t M, int64_t K, const uint16_t* w, int64_t N, double eps,
                     uint32_t* y, double* v, double* sabs) {
    if (M < 0 || K <= 0 || N <= 0 || !(eps >= 0.0)) return -1;
    if (M > 0 && (!x || !w || !y)) return -1;
    double* a = (double*)malloc(sizeof(double) * (size_t)N);
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    if (!a || !s) { free(a); free(s); return -1; }
    for (int64_t i = 0; i < M; ++i) {
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) { a[j] = 0.0; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            const double xv = bio_bf16_to_f64(x[i * K + k]);
            ss = ss + xv * xv;
            for (int64_t j = 0; j < N; ++j) {
                const double p = xv * bio_bf16_to_f64(w[k * N + j]);
                a[j] = a[j] + p;
                s[j] = s[j] + fabs(p);
            }
        }
        const double rms = sqrt(ss / (double)K + eps);
        for (int64_t j = 0; j < N; ++j) {
            const double val = a[j] / rms;
            y[i * N + j] = bio_f64_to_f32(val);
            if (v) v[i * N + j] = val;
            if (sabs) sabs[i * N + j] = s[j] / rms;
        }
    }
    free(a);
    free(s);
    return 0;
}
