"""Pins of the mHC pre-norm projection oracle (``oracle.prenorm_gemm``) to what the mathematics
fixes, not to itself: exact rational arithmetic on small cases (the fp32 rounding of
a / sqrt(ss/K + eps) decided by comparing squares), exact invariance under scaling a row by 2^k
without epsilon, the identity RMSNorm(x) . W = (x . W) / rms(x) against the RMSNorm and GEMM
oracles, torch's rms_norm followed by a matmul in fp64, row decomposition, and planted mistakes
(a mean over K - 1, a dropped epsilon, a transposed W) failing the torch check.  Definition:
"[BI][DSv4] Make mHC tilelang ops batch invariant" (the pre-norm GEMM with its fused RMSNorm)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from exact import bf16_value, f32_bits_of_signed_sqrt

EPS = float(np.float32(1e-6))


def f64(bits):
    return ig.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


@pytest.mark.parametrize("M,K,N,eps", [(3, 8, 4, 0.0), (2, 40, 6, 2.0**-10), (4, 16, 24, 0.25)])
def test_exact_small_cases(M, K, N, eps):
    x = ig.scaled_rows_bf16(3 + K, M, K)
    w = ig.normal_bf16(4 + K, K, N, std=0.02)
    y, v, _ = oracle.prenorm_gemm(x, w, eps)
    for i in range(M):
        xs = [bf16_value(int(b)) for b in x[i]]
        den = sum((t * t for t in xs), Fraction(0)) / K + Fraction(eps)
        for j in range(N):
            a = sum((xs[k] * bf16_value(int(w[k, j])) for k in range(K)), Fraction(0))
            q = a * a / den
            assert int(y.view(np.uint32)[i, j]) == f32_bits_of_signed_sqrt(q, a < 0), (i, j)
            vv = Fraction(float(v[i, j]))
            assert (vv < 0) == (a < 0) and abs(vv * vv - q) <= q * Fraction(1, 2**50)


@pytest.mark.parametrize("k", [-30, -3, 7, 40])
def test_scale_invariance_without_epsilon(k):
    x = ig.scaled_rows_bf16(5, 6, 512)
    w = ig.normal_bf16(6, 512, 24, std=0.02)
    xs = ig.to_bf16_bits(f64(x) * 2.0**k)
    assert np.array_equal(f64(xs), f64(x) * 2.0**k)
    y1, v1, _ = oracle.prenorm_gemm(x, w, 0.0)
    y2, v2, _ = oracle.prenorm_gemm(xs, w, 0.0)
    assert np.array_equal(y1, y2) and np.array_equal(v1, v2)


def test_equals_rmsnorm_then_gemm():
    """(x . W) / rms(x) = RMSNorm(x) . W (weight 1): the RMSNorm oracle's unrounded rows times W
    (the fp64 GEMM oracle) agree with this oracle's values within fp64 rounding."""
    K, N = 1024, 24
    x = ig.scaled_rows_bf16(7, 9, K)
    w = ig.normal_bf16(8, K, N, std=0.02)
    _, v, sabs = oracle.prenorm_gemm(x, w, EPS)
    _, xn = oracle.rmsnorm_bf16(x, np.full(K, 0x3F80, np.uint16), EPS)
    acc, _ = oracle.gemm_f64(xn, f64(w))
    assert np.all(np.abs(acc - v) <= 1e-13 * sabs)


def test_against_torch_fp64():
    K, N = 16384, 24
    x = ig.scaled_rows_bf16(9, 5, K)
    w = ig.normal_bf16(10, K, N, std=0.02)
    _, v, sabs = oracle.prenorm_gemm(x, w, EPS)
    ref = (torch.nn.functional.rms_norm(torch.from_numpy(f64(x)), (K,), eps=EPS) @ torch.from_numpy(f64(w))).numpy()
    assert np.all(np.abs(v - ref) <= 1e-12 * sabs)


def test_row_decomposition():
    x = ig.scaled_rows_bf16(11, 12, 256)
    w = ig.normal_bf16(12, 256, 24, std=0.02)
    y, v, _ = oracle.prenorm_gemm(x, w, EPS)
    for sp in (1, 5, 11):
        ya, va, _ = oracle.prenorm_gemm(x[:sp], w, EPS)
        yb, vb, _ = oracle.prenorm_gemm(x[sp:], w, EPS)
        assert np.array_equal(np.vstack([ya, yb]), y) and np.array_equal(np.vstack([va, vb]), v)


def _mutant(kind, x, w, eps):
    xf, wf = f64(x), f64(w)
    K = x.shape[1]
    ss = np.sum(xf * xf, axis=1, keepdims=True)
    ms = ss / (K - 1) if kind == "mean_over_k_minus_1" else ss / K
    e = 0.0 if kind == "no_epsilon" else eps
    wm = wf.T if kind == "transposed_w" else wf
    return (xf @ wm) / np.sqrt(ms + e)


@pytest.mark.parametrize("kind", ["mean_over_k_minus_1", "no_epsilon", "transposed_w"])
def test_planted_mistakes_fail_the_torch_check(kind):
    K = 64
    x = ig.scaled_rows_bf16(13, 4, K, scales=(2.0**-8, 2.0**-9, 2.0**-10))
    w = ig.normal_bf16(14, K, K, std=0.02)
    eps = 2.0**-18
    _, v, sabs = oracle.prenorm_gemm(x, w, eps)
    ref = (torch.nn.functional.rms_norm(torch.from_numpy(f64(x)), (K,), eps=eps) @ torch.from_numpy(f64(w))).numpy()
    assert np.all(np.abs(v - ref) <= 1e-12 * sabs)
    bad = _mutant(kind, x, w, eps)
    assert not np.all(np.abs(bad - ref) <= 1e-12 * sabs)


def test_tolerance_covers_chunked_fp32_evaluation():
    """The GPU tolerance |y - v| <= TOL_PRENORM_ABS * sabs + 2^-15 |v| covers an fp32 evaluation
    with sequential fma sums over chunks of 512, chunks added in order, at K = 16384."""
    K, N, M = 16384, 24, 6
    x = ig.scaled_rows_bf16(15, M, K)
    w = ig.normal_bf16(16, K, N, std=0.02)
    _, v, sabs = oracle.prenorm_gemm(x, w, EPS)
    xf = ig.bf16_bits_to_f32(x)
    wf = ig.bf16_bits_to_f32(w)
    for i in range(M):
        acc = np.zeros(N, np.float32)
        ss = np.float32(0)
        for c0 in range(0, K, 512):
            pa = np.zeros(N, np.float32)
            ps = np.float32(0)
            for k in range(c0, c0 + 512):
                pa = (pa + xf[i, k] * wf[k]).astype(np.float32)
                ps = np.float32(ps + xf[i, k] * xf[i, k])
            acc = (acc + pa).astype(np.float32)
            ss = np.float32(ss + ps)
        r = np.float32(1) / np.sqrt(np.float32(np.float32(ss / np.float32(K)) + np.float32(EPS)))
        y = (acc * r).astype(np.float64)
        assert np.all(np.abs(y - v[i]) <= oracle.TOL_PRENORM_ABS * sabs[i] + 2.0**-15 * np.abs(v[i]))


def test_bad_arguments_rejected():
    with pytest.raises(ValueError):
        oracle.prenorm_gemm(np.zeros((2, 8), np.uint16), np.zeros((8, 3), np.uint16), -1.0)
    with pytest.raises(ValueError):
        oracle.prenorm_gemm(np.zeros((2, 0), np.uint16), np.zeros((0, 3), np.uint16), 0.0)
