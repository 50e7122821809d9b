"""CPU oracle for the batch-invariant GEMM y = x·W and RMSNorm — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product (``invariant_bi_gemm_gb300``) never does, and the
two share no code: the oracle is plain C (``bi_oracle.c``) built with gcc.

Definition followed ("Batch-invariant matrix multiplication", nondeterminism
article; the row-wise definition y[i] = f(x[i], W) of the batch-invariance issue,
"Problem statement"):

    y[i, j] = round_out( sum_{k ascending} dec(x[i, k]) * dec(w[k, j]) )   (fp64 sum)

with a single round-to-nearest-even to the output dtype, and the absolute sum
S_abs[i, j] = sum_k |dec(x[i, k]) * dec(w[k, j])| returned for the tolerance.

Attention ("Batch-invariant attention", nondeterminism article): for each query token at
position p and head, the fp64 softmax-weighted mean of the values at positions 0..p, rounded
once to bf16, with the unrounded value and the error scales returned for the tolerance.

mHC pre-norm projection ("[BI][DSv4] Make mHC tilelang ops batch invariant"): the projection
x_i . W divided by the root mean square of x_i, in fp64, rounded once to fp32.

RMSNorm ("Batch-invariant RMSNorm", nondeterminism article): for each row,
v[i, j] = (x[i, j] / sqrt(sum_{j ascending} x[i, j]^2 / d + eps)) * g[j] in fp64,
rounded once to bf16; v is returned for the tolerance.

Every function here is pinned by ``tests/test_oracle_*.py`` against exact
rational arithmetic, the pages' worked examples and identities, and library
routines; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

OUT_BF16 = 0
OUT_F32 = 1

_lib = None


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.bio_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.bio_bf16_to_f64.restype = ctypes.c_double
        L.bio_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.bio_e4m3_to_f64.restype = ctypes.c_double
        L.bio_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        L.bio_e8m0_to_f64.restype = ctypes.c_double
        L.bio_f64_to_bf16.argtypes = [ctypes.c_double]
        L.bio_f64_to_bf16.restype = ctypes.c_uint16
        L.bio_f64_to_f32.argtypes = [ctypes.c_double]
        L.bio_f64_to_f32.restype = ctypes.c_uint32
        L.bio_gemm_f64.argtypes = [P, I64, I64, P, I64, P, P]
        L.bio_gemm_f64.restype = ctypes.c_int
        L.bio_gemm_bf16.argtypes = [P, I64, I64, P, I64, P, I64, ctypes.c_int, P, P, P]
        L.bio_gemm_bf16.restype = ctypes.c_int
        L.bio_gemm_mxfp8.argtypes = [P, P, I64, I64, P, P, I64, P, I64, P, P, P]
        L.bio_gemm_mxfp8.restype = ctypes.c_int
        L.bio_rmsnorm_bf16.argtypes = [P, I64, I64, P, ctypes.c_double, P, I64, P, P]
        L.bio_rmsnorm_bf16.restype = ctypes.c_int
        L.bio_attention_bf16.argtypes = [P, I64, I64, I64, P, P, P, P, I64, I64, I64, P, I64, I64,
                                         ctypes.c_double, P, P, P, P]
        L.bio_attention_bf16.restype = ctypes.c_int
        L.bio_prenorm_gemm.argtypes = [P, I64, I64, P, I64, ctypes.c_double, P, P, P]
        L.bio_prenorm_gemm.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, int(r.shape[0])


def gemm_f64(x: np.ndarray, w: np.ndarray):
    """fp64 inputs; returns (acc, sabs) fp64 [M, N] without output rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    M, K = x.shape
    K2, N = w.shape
    assert K == K2
    acc = np.empty((M, N), np.float64)
    sabs = np.empty((M, N), np.float64)
    rc = lib().bio_gemm_f64(_ptr(x), M, K, _ptr(w), N, _ptr(acc), _ptr(sabs))
    if rc:
        raise ValueError("bio_gemm_f64 rejected its arguments")
    return acc, sabs


def gemm_bf16(x: np.ndarray, w: np.ndarray, out: str = "bf16", rows=None):
    """x uint16[M,K], w uint16[K,N] (bf16 patterns).

    Returns (y, acc, sabs): y uint16 bf16 patterns or float32 values [R, N] where R is
    len(rows) (the listed rows of x, in that order) or M; acc and sabs fp64 [R, N].
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    M, K = x.shape
    K2, N = w.shape
    assert K == K2
    r, R = _rows_arg(rows, M)
    if out == "bf16":
        y = np.empty((R, N), np.uint16)
        kind = OUT_BF16
    elif out == "f32":
        y = np.empty((R, N), np.uint32)
        kind = OUT_F32
    else:
        raise ValueError(out)
    acc = np.empty((R, N), np.float64)
    sabs = np.empty((R, N), np.float64)
    rc = lib().bio_gemm_bf16(_ptr(x), M, K, _ptr(w), N, _ptr(r), R, kind, _ptr(y), _ptr(acc), _ptr(sabs))
    if rc:
        raise ValueError("bio_gemm_bf16 rejected its arguments")
    if out == "f32":
        y = y.view(np.float32)
    return y, acc, sabs


def gemm_mxfp8(x, sx, w, sw, rows=None):
    """x uint8[M,K] E4M3, sx uint8[M,K/32] E8M0, w uint8[K,N] E4M3, sw uint8[K/32,N] E8M0.

    Returns (y bf16 patterns uint16 [R, N], acc, sabs) as gemm_bf16.
    """
    x = np.ascontiguousarray(x, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.uint8)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    sw = np.ascontiguousarray(sw, dtype=np.uint8)
    M, K = x.shape
    K2, N = w.shape
    assert K == K2 and sx.shape == (M, K // 32) and sw.shape == (K // 32, N)
    r, R = _rows_arg(rows, M)
    y = np.empty((R, N), np.uint16)
    acc = np.empty((R, N), np.float64)
    sabs = np.empty((R, N), np.float64)
    rc = lib().bio_gemm_mxfp8(_ptr(x), _ptr(sx), M, K, _ptr(w), _ptr(sw), N, _ptr(r), R,
                              _ptr(y), _ptr(acc), _ptr(sabs))
    if rc:
        raise ValueError("bio_gemm_mxfp8 rejected its arguments")
    return y, acc, sabs


def rmsnorm_bf16(x: np.ndarray, g: np.ndarray, eps: float, rows=None):
    """RMSNorm of bf16 rows ("Batch-invariant RMSNorm", nondeterminism article).

    x uint16[M, d], g uint16[d] (bf16 patterns), eps the fp32 value the GPU adds, passed as
    a double.  Returns (y uint16 bf16 patterns [R, d], v fp64 [R, d] unrounded).
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    g = np.ascontiguousarray(g, dtype=np.uint16)
    M, d = x.shape
    assert g.shape == (d,)
    r, R = _rows_arg(rows, M)
    y = np.empty((R, d), np.uint16)
    v = np.empty((R, d), np.float64)
    rc = lib().bio_rmsnorm_bf16(_ptr(x), M, d, _ptr(g), float(eps), _ptr(r), R, _ptr(y), _ptr(v))
    if rc:
        raise ValueError("bio_rmsnorm_bf16 rejected its arguments")
    return y, v


def attention_bf16(q, q_seq, q_pos, k_cache, v_cache, page_table, scale):
    """Causal attention over a paged KV cache ("Batch-invariant attention", nondeterminism
    article).  q uint16[T, Hq, D]; q_seq, q_pos int32[T]; k_cache, v_cache uint16[P, page, Hkv, D];
    page_table int32[B, max_pages]; scale the fp32 value the GPU uses, passed as a double.

    Returns (o uint16 [T, Hq, D], v fp64 [T, Hq, D], a fp64 [T, Hq, D], e fp64 [T, Hq]).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    q_seq = np.ascontiguousarray(q_seq, dtype=np.int32)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int32)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    T, Hq, D = q.shape
    P_, page, Hkv, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape and q_seq.shape == (T,) and q_pos.shape == (T,)
    B, max_pages = page_table.shape
    o = np.empty((T, Hq, D), np.uint16)
    v = np.empty((T, Hq, D), np.float64)
    a = np.empty((T, Hq, D), np.float64)
    e = np.empty((T, Hq), np.float64)
    rc = lib().bio_attention_bf16(_ptr(q), T, Hq, D, _ptr(q_seq), _ptr(q_pos), _ptr(k_cache), _ptr(v_cache),
                                  P_, page, Hkv, _ptr(page_table), B, max_pages, float(scale),
                                  _ptr(o), _ptr(v), _ptr(a), _ptr(e))
    if rc:
        raise ValueError("bio_attention_bf16 rejected its arguments")
    return o, v, a, e


def prenorm_gemm(x: np.ndarray, w: np.ndarray, eps: float):
    """mHC pre-norm projection ("[BI][DSv4] Make mHC tilelang ops batch invariant"): RMSNorm of
    each row of x (no weight) times W, in fp64, rounded once to fp32.  x uint16[M, K], w
    uint16[K, N] (bf16 patterns); eps the fp32 value the GPU adds, passed as a double.

    Returns (y float32 [M, N], v fp64 [M, N] unrounded, sabs fp64 [M, N] = sum|x w| / rms).
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    M, K = x.shape
    K2, N = w.shape
    assert K == K2
    y = np.empty((M, N), np.uint32)
    v = np.empty((M, N), np.float64)
    sabs = np.empty((M, N), np.float64)
    rc = lib().bio_prenorm_gemm(_ptr(x), M, K, _ptr(w), N, float(eps), _ptr(y), _ptr(v), _ptr(sabs))
    if rc:
        raise ValueError("bio_prenorm_gemm rejected its arguments")
    return y.view(np.float32), v, sabs


# mHC pre-norm projection (fp32 out): |y - v| <= TOL_PRENORM_ABS * sabs + 2^-15 |v|.  A split of K
# into chunks of at most 512 summed in order, chunks merged in order, bounds the fp32 error of the
# projection by gamma_{512 + S}(2^-24) sum|x w| (S <= 64 chunks for K <= 32768: 3.4e-5); the root
# mean square adds at most 2^-16 relative (a sum of positive squares under the same bound, halved
# by the square root, plus the division and the reciprocal square root), the product and the
# fp32 rounding 2^-23 more.
TOL_PRENORM_ABS = 4e-5


def bf16_to_f64(b) -> float:
    return lib().bio_bf16_to_f64(int(b))


def e4m3_to_f64(c) -> float:
    return lib().bio_e4m3_to_f64(int(c))


def e8m0_to_f64(e) -> float:
    return lib().bio_e8m0_to_f64(int(e))


def f64_to_bf16(v: float) -> int:
    return int(lib().bio_f64_to_bf16(float(v)))


def f64_to_f32_bits(v: float) -> int:
    return int(lib().bio_f64_to_f32(float(v)))


def bf16_array_to_f64(b: np.ndarray) -> np.ndarray:
    """Vector decode through the oracle's own scalar decoder semantics (bits << 16)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# Tolerances from the unit roundoffs u(bf16) = 2^-8 and u(fp32) = 2^-24 of the
# nondeterminism article ("Quantifying with unit roundoff"), as fixed for this GEMM:
# bf16 output |y - y_ref| <= 4 * 2^-8 * S_abs, fp32 output |y - y_ref| <= 1e-5 * S_abs.
TOL_BF16 = 4.0 * 2.0**-8
TOL_F32 = 1e-5


def tolerance_violations(y_gpu_f64: np.ndarray, y_ref_f64: np.ndarray, sabs: np.ndarray, tol: float):
    """Return (count, max ratio |y - y_ref| / S_abs) under the rule |y - y_ref| <= tol * S_abs."""
    d = np.abs(y_gpu_f64 - y_ref_f64)
    bad = ~(d <= tol * sabs)   # NaN counts as a violation
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(sabs > 0, d / sabs, np.where(d == 0, 0.0, np.inf))
    return int(bad.sum()), float(np.nanmax(ratio)) if ratio.size else 0.0


# RMSNorm (bf16 out): |y - v| <= (2^-8 + 2^-16) * |v| with v the oracle's unrounded fp64
# value.  2^-8 is the bf16 rounding of the output; 2^-16 bounds the relative error of the fp32
# computation before that rounding (sum of at most 136 positive squares, one division, one
# reciprocal square root of at most 2 ulp, two products: below 1e-5 for d <= 16384).
TOL_RMSNORM_REL = 2.0**-8 + 2.0**-16


def attention_tolerance(v: np.ndarray, a: np.ndarray, e: np.ndarray, D: int, L: np.ndarray) -> np.ndarray:
    """Per-element bound on |o - v| for an fp32 evaluation of the attention rounded to bf16:

        2^-8 |v|  +  (4 (D + 8) u e + 2 (L + 32) u) a,      u = 2^-24

    2^-8 |v| is the bf16 rounding of the output.  The second term covers fp32 arithmetic before
    it: a score is a D-term fp32 dot product times the scale, so its absolute error is at most
    about (D + 4) u e (e = max_j scale sum_i |q_i k_ji|); an error d in the exponent of a weight
    changes the weight by a factor e^d, and the weights enter both the weighted sum and its
    normaliser (hence 2 x 2 (D + 8) u e, which also absorbs the maximum's subtraction, exp's few
    ulp and the rescaling of split partials); the two sums over L = p + 1 positions of positive
    weights (times |v| in the numerator) add at most (L + 32) u a each in any fixed order.
    a = sum_j w_j |v_j| / sum_j w_j bounds |v| and is the natural scale of these errors.
    v, a [T, Hq, D]; e [T, Hq]; L [T] (key count of each query token)."""
    u = 2.0**-24
    L = np.asarray(L, dtype=np.float64)[:, None, None]
    return 2.0**-8 * np.abs(v) + (4.0 * (D + 8) * u * e[:, :, None] + 2.0 * (L + 32) * u) * a


__all__ = [
    "prenorm_gemm", "TOL_PRENORM_ABS",
    "attention_tolerance", "attention_bf16", "rmsnorm_bf16", "TOL_RMSNORM_REL",
    "gemm_f64", "gemm_bf16", "gemm_mxfp8", "bf16_to_f64", "e4m3_to_f64", "e8m0_to_f64",
    "f64_to_bf16", "f64_to_f32_bits", "bf16_array_to_f64", "TOL_BF16", "TOL_F32",
    "tolerance_violations", "lib",
]
