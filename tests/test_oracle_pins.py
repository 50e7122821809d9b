"""Pins of the CPU oracle against facts fixed outside it.

Each test ties one part of the oracle to something it could get wrong: the
decoders and the output rounding to exact rational arithmetic; the dot product
to brute force; the summation order to the pages' worked examples; the
row-wise definition to the row-decomposition identity; the error model to the
gamma_n and log2 n bounds.  A dropped term, a wrong sign, a transposed operand,
a reversed k order or a double rounding each fails at least one of them.
"""
import itertools
import math
import random
import sys
from fractions import Fraction

import numpy as np
import pytest

import inputgen as ig
import oracle
from exact import (bf16_value, e4m3_value, e8m0_value, gamma, round_to_binary,
                   to_bf16_bits_exact, to_f32_bits_exact)
from conftest import read_golden


# ----------------------------------------------------------------- decoders

def test_bf16_decode_all_finite_patterns():
    for b in range(0, 0x10000, 7):
        if (b >> 7) & 0xFF == 0xFF:
            continue
        assert Fraction(oracle.bf16_to_f64(b)) == bf16_value(b), hex(b)
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC000) == -2.0
    assert oracle.bf16_to_f64(0x0001) == 2.0**-133
    assert oracle.bf16_to_f64(0x7F7F) == (2 - 2**-7) * 2.0**127
    assert math.isinf(oracle.bf16_to_f64(0x7F80))


def test_e4m3_decode_all_codes():
    for c in range(256):
        v = oracle.e4m3_to_f64(c)
        if (c & 0x7F) == 0x7F:
            assert math.isnan(v)
            continue
        assert Fraction(v) == e4m3_value(c), hex(c)
    # OCP E4M3FN landmarks: max normal, min normal, min subnormal, one.
    assert oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x08) == 2.0**-6
    assert oracle.e4m3_to_f64(0x01) == 2.0**-9
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0xB8) == -1.0


def test_e8m0_decode():
    for e in range(255):
        assert Fraction(oracle.e8m0_to_f64(e)) == e8m0_value(e)
    assert oracle.e8m0_to_f64(127) == 1.0
    assert math.isnan(oracle.e8m0_to_f64(255))


# ----------------------------------------------------------- output rounding

def _random_doubles(n, seed):
    rng = random.Random(seed)
    out = []
    for _ in range(n):
        e = rng.randint(-140, 130)
        m = rng.getrandbits(52)
        v = math.ldexp(1.0 + m * 2.0**-52, e)
        out.append(-v if rng.random() < 0.5 else v)
    return out


def test_bf16_rounding_matches_exact_rne():
    cases = _random_doubles(20000, 1)
    # ties and near-ties in every regime, overflow edge, subnormals
    for base in (1.0, 3.0, 2.0**-126, 2.0**-130, 2.0**100, (2 - 2**-7) * 2.0**127):
        q = 2.0 ** (math.floor(math.log2(base)) - 7) if base >= 2.0**-126 else 2.0**-133
        for k in range(-3, 4):
            for d in (-1e-3, 0.0, 1e-3):
                cases.append(base + (k + 0.5 + d) * q)
    cases += [0.0, -0.0, 2.0**-134, 2.0**-134 * 1.0000001, 3 * 2.0**-134, 1e-300, -1e-300]
    for v in cases:
        want = (0x8000 if math.copysign(1.0, v) < 0 else 0) if v == 0 else to_bf16_bits_exact(Fraction(v))
        assert oracle.f64_to_bf16(v) == want, repr(v)


def test_bf16_rounding_textbook_ties():
    assert oracle.f64_to_bf16(1.0 + 2.0**-8) == 0x3F80          # tie -> even (down)
    assert oracle.f64_to_bf16(1.0 + 3 * 2.0**-8) == 0x3F82      # tie -> even (up)
    assert oracle.f64_to_bf16(1.0 + 2.0**-8 + 2.0**-40) == 0x3F81
    assert oracle.f64_to_bf16(-(1.0 + 2.0**-8)) == 0xBF80
    assert oracle.f64_to_bf16(3.4e38) == 0x7F80                 # rounds past max -> inf
    assert oracle.f64_to_bf16(float("nan")) & 0x7FC0 == 0x7FC0


def test_f32_rounding_matches_exact_and_numpy():
    cases = _random_doubles(20000, 2)
    for v in cases:
        bits = oracle.f64_to_f32_bits(v)
        assert bits == to_f32_bits_exact(Fraction(v)), repr(v)
        with np.errstate(over="ignore"):
            assert bits == int(np.array([v], np.float64).astype(np.float32).view(np.uint32)[0])


# --------------------------------------------------------- brute force GEMM

def _exact_dot_rows(xv, wv):
    M, K = len(xv), len(xv[0])
    N = len(wv[0])
    return [[sum((xv[i][k] * wv[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
            for i in range(M)]


@pytest.mark.parametrize("M,K,N,seed", [(1, 1, 1, 5), (3, 7, 2, 6), (4, 64, 4, 7), (2, 33, 3, 8), (4, 16, 1, 9)])
def test_brute_force_bf16_exact(M, K, N, seed):
    x = ig.normal_bf16(seed, M, K)
    w = ig.normal_bf16(seed + 100, K, N, std=0.05)
    xv = [[bf16_value(int(b)) for b in row] for row in x]
    wv = [[bf16_value(int(b)) for b in row] for row in w]
    ex = _exact_dot_rows(xv, wv)
    yb, acc, sabs = oracle.gemm_bf16(x, w, "bf16")
    yf, acc2, _ = oracle.gemm_bf16(x, w, "f32")
    assert np.array_equal(acc, acc2)
    for i in range(M):
        for j in range(N):
            # N(0,1) bf16 inputs keep every partial sum within 53 bits: the fp64 sum is exact.
            assert Fraction(acc[i, j]) == ex[i][j]
            assert Fraction(sabs[i, j]) == sum(abs(xv[i][k] * wv[k][j]) for k in range(K))
            assert int(yb[i, j]) == to_bf16_bits_exact(ex[i][j])
            assert int(yf.view(np.uint32)[i, j]) == to_f32_bits_exact(ex[i][j])


def test_brute_force_wide_range_within_fp64_bound():
    """Exponents over +-60 force the fp64 running sum to round: the oracle stays within
    gamma_{K-1}(2^-53) * S_abs of the exact sum, and its bf16 output equals the exactly
    rounded value except where the exact sum lies within that error of a rounding boundary."""
    rng = random.Random(11)
    M, K, N = 3, 48, 3
    x = np.array([[(rng.randint(67, 187) << 7) | rng.getrandbits(7) |
                   (0x8000 if rng.random() < .5 else 0) for _ in range(K)] for _ in range(M)], np.uint16)
    w = np.array([[(rng.randint(100, 154) << 7) | rng.getrandbits(7) | (0x8000 if rng.random() < .5 else 0)
                   for _ in range(N)] for _ in range(K)], np.uint16)
    xv = [[bf16_value(int(b)) for b in row] for row in x]
    wv = [[bf16_value(int(b)) for b in row] for row in w]
    ex = _exact_dot_rows(xv, wv)
    yb, acc, sabs = oracle.gemm_bf16(x, w, "bf16")
    g = gamma(K - 1, 2.0**-53)
    near_boundary = 0
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(acc[i, j]) - ex[i][j])
            assert err <= Fraction(g) * Fraction(sabs[i, j])
            if int(yb[i, j]) != to_bf16_bits_exact(ex[i][j]):
                lo = to_bf16_bits_exact(ex[i][j] - err)
                hi = to_bf16_bits_exact(ex[i][j] + err)
                assert lo != hi, "output differs although no rounding boundary is within the fp64 error"
                near_boundary += 1
    assert near_boundary <= 1


def test_brute_force_mxfp8_exact():
    M, K, N = 3, 96, 4
    x = ig.normal_e4m3(21, M, K)
    w = ig.normal_e4m3(22, K, N)
    sx = ig.e8m0_scales("VAR", 23, M, K // 32)
    sw = ig.e8m0_scales("VAR", 24, K // 32, N)
    y, acc, sabs = oracle.gemm_mxfp8(x, sx, w, sw)
    for i in range(M):
        for j in range(N):
            ex = sum((e4m3_value(int(x[i, k])) * e8m0_value(int(sx[i, k // 32])) *
                      e4m3_value(int(w[k, j])) * e8m0_value(int(sw[k // 32, j])) for k in range(K)),
                     Fraction(0))
            assert Fraction(acc[i, j]) == ex
            assert int(y[i, j]) == to_bf16_bits_exact(ex)


def test_planted_transpose_is_caught():
    """The brute-force pin separates y = x·W from y = x·W^T on a square W (a plausible
    operand mix-up): the two differ in the oracle's own output."""
    x = ig.normal_bf16(31, 2, 8)
    w = ig.normal_bf16(32, 8, 8)
    y1, _, _ = oracle.gemm_bf16(x, w, "f32")
    y2, _, _ = oracle.gemm_bf16(x, np.ascontiguousarray(w.T), "f32")
    assert not np.array_equal(y1, y2)
    xv = [[bf16_value(int(b)) for b in row] for row in x]
    wv = [[bf16_value(int(b)) for b in row] for row in w]
    ex = _exact_dot_rows(xv, wv)
    assert all(int(y1.view(np.uint32)[i, j]) == to_f32_bits_exact(ex[i][j]) for i in range(2) for j in range(8))


# ------------------------------------------------------ identities of the pages

def test_row_decomposition_identity():
    """[A; B] C = [A C; B C] ("Batch invariance", nondeterminism article), bitwise,
    for the page's split at k and for every split point of a small batch."""
    x = ig.normal_bf16(41, 12, 96)
    w = ig.normal_bf16(42, 96, 40, std=0.02)
    for out in ("bf16", "f32"):
        full, acc, _ = oracle.gemm_bf16(x, w, out)
        for k in range(0, 13):
            top, acc_t, _ = oracle.gemm_bf16(x[:k], w, out)
            bot, acc_b, _ = oracle.gemm_bf16(x[k:], w, out)
            assert np.array_equal(np.concatenate([top, bot]).view(np.uint8), full.view(np.uint8))
            assert np.array_equal(np.concatenate([acc_t, acc_b]), acc)
    # row subset interface equals full-matrix rows
    sub, _, _ = oracle.gemm_bf16(x, w, "bf16", rows=[11, 0, 5])
    assert np.array_equal(sub, full_bf16 := oracle.gemm_bf16(x, w, "bf16")[0][[11, 0, 5]])
    assert full_bf16.shape == (3, 40)


def test_nonassociativity_example_pins_ascending_k():
    g = read_golden("nonassociativity.txt")
    assert float(g["(0.1 + 1e20) - 1e20"]) == 0.0 and float(g["0.1 + (1e20 - 1e20)"]) == 0.1
    ones = np.ones((3, 1))
    a, _ = oracle.gemm_f64(np.array([[0.1, 1e20, -1e20]]), ones)
    b, _ = oracle.gemm_f64(np.array([[1e20, -1e20, 0.1]]), ones)
    assert a[0, 0] == 0.0          # ((0.1 + 1e20) - 1e20): summed in ascending k
    assert b[0, 0] == 0.1          # ((1e20 - 1e20) + 0.1)


def _seq_sum_exact_rne(values):
    """Left-to-right fp64 sum with every add rounded exactly (rational arithmetic + RNE)."""
    s = Fraction(0)
    for v in values:
        sign, units, qe = round_to_binary(s + Fraction(v), 53, -1022, 1023)
        s = sign * Fraction(units) * (Fraction(2) ** qe)
    return float(s)


def test_eight_value_example():
    """Worked example of the nondeterminism article ("Quantifying with unit roundoff").

    The oracle's fp64 sums of the page's 10000 shuffled orders equal sums computed with
    exact rational arithmetic and one round-to-nearest-even per add, in ascending k; the
    exact sum is 0, every rounded sum lies within gamma_7 * sum|v|, and the two extremes
    the page prints occur.  (The page's count of 102 distinct values comes from CPython's
    built-in sum(), which is compensated since 3.12; plain left-to-right summation, the
    oracle's definition, gives more distinct values.  The last check confirms that reading,
    with the page's list as typed: 1 and -1 are Python integers there.)
    """
    g = read_golden("eight_values.txt")
    vals = [float(t) for t in g["values"].split()]
    assert sum(Fraction(v) for v in vals) == int(g["exact_sum"]) == 0
    rng = random.Random(int(g["seed"]))
    order = list(vals)
    rows = []
    for _ in range(int(g["shuffles"])):
        rng.shuffle(order)
        rows.append(list(order))
    acc, sabs = oracle.gemm_f64(np.array(rows), np.ones((8, 1)))
    s = acc[:, 0]
    for r, got in zip(rows[:2000], s[:2000]):
        assert got == _seq_sum_exact_rne(r)
    uniq = set(s.tolist())
    assert len(uniq) > 1                               # order changes the result
    assert float(g["min_result"]) in uniq and float(g["max_result"]) in uniq
    assert np.all(np.abs(s) <= gamma(7, 2.0**-53) * sabs[:, 0])
    # all 8! orders
    perms = np.array(list(itertools.permutations(vals)))
    acc, sabs = oracle.gemm_f64(perms, np.ones((8, 1)))
    assert np.all(np.abs(acc[:, 0]) <= gamma(7, 2.0**-53) * sabs[:, 0])
    if sys.version_info >= (3, 12):
        # the page's list holds the integers 1 and -1 beside floats, as typed
        typed = [int(t) if t.lstrip("-").isdigit() else float(t) for t in g["values"].split()]
        rng = random.Random(int(g["seed"]))
        order = list(typed)
        builtin = set()
        for _ in range(int(g["shuffles"])):
            rng.shuffle(order)
            builtin.add(sum(order))
        assert len(builtin) == int(g["distinct_results"])


def test_unit_roundoff_table():
    g = read_golden("unit_roundoff.txt")
    for name, p, u_printed in g["_rows"]:
        u = 2.0 ** -int(p)
        assert float(f"{u:.2e}") == float(u_printed), name
    # the tolerances are built on these: bf16 u = 2^-8, fp32 u = 2^-24
    assert oracle.TOL_BF16 == 4 * 2.0**-8


def _pairwise_f32(v):
    """Pure pairwise (tree) sum in fp32: adjacent pairs added level by level."""
    a = np.asarray(v, np.float32)
    depth = 0
    while a.size > 1:
        if a.size % 2:
            a = np.concatenate([a, np.zeros(1, np.float32)])
        a = (a[0::2] + a[1::2]).astype(np.float32)
        depth += 1
    return float(a[0]), depth


@pytest.mark.parametrize("logn", [4, 8, 12, 16])
def test_summation_error_bounds(logn):
    """Sequential-sum bound gamma_{n-1} * sum|x| and tree-sum bound with depth ceil(log2 n)
    ("Quantifying with unit roundoff", nondeterminism article), using the oracle's fp64
    sum, itself within gamma_{n-1}(2^-53) of the exact sum, as the reference."""
    n = 2**logn + 3
    x = (ig.normal(50 + logn, 0, n) * np.exp(ig.normal(60 + logn, 0, n))).astype(np.float32)
    exact = sum((Fraction(float(t)) for t in x), Fraction(0))
    acc, sabs = oracle.gemm_f64(x.astype(np.float64)[None, :], np.ones((n, 1)))
    assert abs(Fraction(acc[0, 0]) - exact) <= Fraction(gamma(n - 1, 2.0**-53)) * Fraction(sabs[0, 0])
    S = float(sabs[0, 0])
    seq = float(np.cumsum(x, dtype=np.float32)[-1])          # left-to-right fp32
    assert abs(Fraction(seq) - exact) <= Fraction(gamma(n - 1, 2.0**-24) * S)
    tree, depth = _pairwise_f32(x)
    assert depth == math.ceil(math.log2(n))
    assert abs(Fraction(tree) - exact) <= Fraction(gamma(depth, 2.0**-24) * S)
    # the page prints the first-order form ceil(log2 n) * u; the rigorous gamma form is used above
    assert gamma(depth, 2.0**-24) >= depth * 2.0**-24


def test_tolerance_covers_fp32_accumulation_then_bf16_rounding():
    """bf16-out tolerance 4*2^-8*S_abs >= gamma_{K-1}(2^-24)*S_abs + 2^-8*|s| for the
    K of every workload (K <= 16384), so any fp32 summation order passes it."""
    for K in (128, 256, 2048, 4096, 16384):
        assert gamma(K - 1, 2.0**-24) + 2.0**-8 <= oracle.TOL_BF16


# -------------------------------------------------------------- special cases

def test_identity_and_one_hot_rows():
    K, N = 64, 24
    w = ig.normal_bf16(71, K, N)
    eye = np.zeros((K, K), np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3F80
    y, _, _ = oracle.gemm_bf16(eye, w, "bf16")
    assert np.array_equal(y, w)                              # I·W = W, exactly representable
    # one non-zero per row: a gather of scaled W rows
    x = np.zeros((5, K), np.uint16)
    idx = [3, 0, 63, 17, 3]
    x[np.arange(5), idx] = 0x4000                            # 2.0
    yf, _, _ = oracle.gemm_bf16(x, w, "f32")
    wf = oracle.bf16_array_to_f64(w)
    assert np.array_equal(yf.astype(np.float64), 2.0 * wf[idx])


def test_mxfp8_identity_scales_equal_bf16_path():
    """With E8M0 = 127 (2^0) the MXFP8 GEMM is the bf16 GEMM of the decoded E4M3 values
    (every E4M3 value is a bf16 value), bit for bit; a K-varying scale equals pre-scaling."""
    M, K, N = 4, 128, 40
    x = ig.normal_e4m3(81, M, K)
    w = ig.normal_e4m3(82, K, N)
    sx1 = ig.e8m0_scales("ID", 0, M, K // 32)
    sw1 = ig.e8m0_scales("ID", 0, K // 32, N)
    y8, acc8, _ = oracle.gemm_mxfp8(x, sx1, w, sw1)
    xb = np.array([[to_bf16_bits_exact(e4m3_value(int(c))) for c in r] for r in x], np.uint16)
    wb = np.array([[to_bf16_bits_exact(e4m3_value(int(c))) for c in r] for r in w], np.uint16)
    yb, accb, _ = oracle.gemm_bf16(xb, wb, "bf16")
    assert np.array_equal(y8, yb) and np.array_equal(acc8, accb)
    sx = ig.e8m0_scales("VAR", 83, M, K // 32)
    sw = ig.e8m0_scales("VAR", 84, K // 32, N)
    y8v, acc8v, _ = oracle.gemm_mxfp8(x, sx, w, sw)
    xs = np.array([[to_bf16_bits_exact(e4m3_value(int(x[i, k])) * e8m0_value(int(sx[i, k // 32])))
                    for k in range(K)] for i in range(M)], np.uint16)
    ws = np.array([[to_bf16_bits_exact(e4m3_value(int(w[k, j])) * e8m0_value(int(sw[k // 32, j])))
                    for j in range(N)] for k in range(K)], np.uint16)
    ybv, accbv, _ = oracle.gemm_bf16(xs, ws, "bf16")
    assert np.array_equal(y8v, ybv) and np.array_equal(acc8v, accbv)
    # a uniform power-of-two row scale scales the exact result (no under/overflow here)
    sx2 = sx1.copy()
    sx2[1, :] = 127 + 3
    _, acc8s, _ = oracle.gemm_mxfp8(x, sx2, w, sw1)
    assert np.array_equal(acc8s[1], acc8[1] * 8.0) and np.array_equal(acc8s[0], acc8[0])


def test_against_library_matmul():
    """numpy's fp64 matmul (another summation order) agrees within gamma_K(2^-53)*S_abs."""
    x = ig.normal_bf16(91, 33, 300)
    w = ig.normal_bf16(92, 300, 70, std=0.02)
    _, acc, sabs = oracle.gemm_bf16(x, w, "f32")
    ref = oracle.bf16_array_to_f64(x) @ oracle.bf16_array_to_f64(w)
    assert np.all(np.abs(ref - acc) <= gamma(300, 2.0**-53) * sabs)
    assert np.allclose(sabs, np.abs(oracle.bf16_array_to_f64(x)) @ np.abs(oracle.bf16_array_to_f64(w)),
                       rtol=1e-12, atol=0)


def test_linspace_rows_are_independent():
    """The linspace stress inputs ("Batch invariance", nondeterminism article) at reduced
    size: the oracle's row 0 of the full product equals the product of row 0 alone."""
    a = ig.linspace_bf16(-1000, 1000, 16, 256)
    b = ig.linspace_bf16(-1000, 1000, 256, 256)
    full, _, _ = oracle.gemm_bf16(a, b, "f32")
    one, _, _ = oracle.gemm_bf16(a[:1], b, "f32")
    assert np.array_equal(full[:1].view(np.uint32), one.view(np.uint32))


def test_bad_arguments_rejected():
    L = oracle.lib()
    assert L.bio_gemm_bf16(None, 2, 2, None, 2, None, 0, 0, None, None, None) == -1
    assert L.bio_gemm_mxfp8(None, None, 1, 33, None, None, 1, None, 0, None, None, None) == -1
    x = ig.normal_bf16(1, 2, 4)
    w = ig.normal_bf16(2, 4, 2)
    with pytest.raises(ValueError):
        oracle.gemm_bf16(x, w, "bf16", rows=[2])


def test_oracle_rows_helper_matches_one_call():
    """The GPU tests spread large oracle calls over host threads (tests/gpu_util.py:oracle_rows);
    the pieces must come back in the order of the requested rows, equal to one call."""
    import gpu_util
    x = ig.normal_bf16(ig.SEED_X, 40, 64)
    w = ig.normal_bf16(ig.SEED_W, 64, 24)
    rows = [5, 0, 39, 12, 7, 3, 5]
    one = oracle.gemm_bf16(x, w, "f32", rows=rows)
    for chunks in (1, 3, 7):
        got = gpu_util.oracle_rows(lambda r: oracle.gemm_bf16(x, w, "f32", rows=r), rows, chunks=chunks)
        assert all(np.array_equal(a, b) for a, b in zip(one, got))
