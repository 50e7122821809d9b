"""Pins of the RMSNorm oracle (``oracle.rmsnorm_bf16``) to what the mathematics fixes, not to
itself: exact rational arithmetic on short rows (the rounding of a square root decided by
comparing squares), closed forms, exact scale invariance, row decomposition, the weight's
column index, the unit mean square of the normalised row, and torch's own ``rms_norm`` in
fp64.  Planted mistakes (a mean over d - 1, a dropped epsilon, a reversed weight) are shown
to fail the exact check.  Definition: "Batch-invariant RMSNorm", nondeterminism article."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from exact import bf16_bits_of_signed_sqrt, bf16_value

EPS_CASES = [0.0, 2.0**-20, float(np.float32(1e-6)), 0.0625]


def _exact(xb: np.ndarray, gb: np.ndarray, eps: float):
    """Per element: (exact bf16 bits, q = v^2 as a Fraction, sign of v)."""
    xs = [bf16_value(int(b)) for b in xb]
    gs = [bf16_value(int(b)) for b in gb]
    den = sum((v * v for v in xs), Fraction(0)) / len(xs) + Fraction(eps)
    out = []
    for xv, gv in zip(xs, gs):
        p = xv * gv
        q = p * p / den
        out.append((bf16_bits_of_signed_sqrt(q, p < 0), q, p < 0))
    return out


def _agrees_exactly(y: np.ndarray, v: np.ndarray, x: np.ndarray, g: np.ndarray, eps: float) -> bool:
    """y must be the exact RNE of the true value; v within 2^-50 of it (fp64 arithmetic)."""
    for i in range(x.shape[0]):
        for j, (bits, q, neg) in enumerate(_exact(x[i], g, eps)):
            if int(y[i, j]) != bits:
                return False
            vv = Fraction(float(v[i, j]))
            if q == 0:
                if vv != 0:
                    return False
                continue
            if (vv < 0) != neg or abs(vv * vv - q) > q * Fraction(1, 2**50):
                return False
    return True


def _rows(seed: int, m: int, d: int, lo: int = -12, hi: int = 12) -> np.ndarray:
    """m bf16 rows of N(0, 1) values, each row scaled by its own power of two in [2^lo, 2^hi]."""
    f = ig.bf16_bits_to_f32(ig.normal_bf16(seed, m, d)).astype(np.float64)
    e = ig.uniform_int(seed + 1000, 0, m, lo, hi).astype(np.float64)
    return ig.to_bf16_bits(f * np.exp2(e)[:, None])


@pytest.mark.parametrize("d", [1, 2, 3, 7, 16, 40])
@pytest.mark.parametrize("eps", EPS_CASES)
def test_exact_short_rows(d, eps):
    x = _rows(11 + d, 4, d)
    g = ig.rmsnorm_weight_bf16(21 + d, d)
    y, v = oracle.rmsnorm_bf16(x, g, eps)
    assert _agrees_exactly(y, v, x, g, eps)


def test_constant_row_closed_forms():
    """Row of d equal values c, weight 1: v = c / sqrt(c^2 + eps).  With c = 1/2, eps = 0 every
    value is exactly 1; with eps = 3/4 exactly 1/2 (ms + eps = 1).  A mean over d - 1, or any
    change to the count, moves v off these exact values."""
    d = 4096
    x = np.full((1, d), 0x3F00, np.uint16)               # 0.5
    g = np.full(d, 0x3F80, np.uint16)                     # 1.0
    y, v = oracle.rmsnorm_bf16(x, g, 0.0)
    assert np.all(v == 1.0) and np.all(y == 0x3F80)
    y, v = oracle.rmsnorm_bf16(x, g, 0.75)
    assert np.all(v == 0.5) and np.all(y == 0x3F00)
    # c = 1/2, eps = 1/4: v = 0.5 / sqrt(0.5) = sqrt(1/2), its bf16 rounding decided exactly
    y, v = oracle.rmsnorm_bf16(x, g, 0.25)
    assert np.all(y == bf16_bits_of_signed_sqrt(Fraction(1, 2), False))
    assert abs(v[0, 0] - 2.0**-0.5) <= 2.0**-52
    # negative constant: sign carried through
    y, v = oracle.rmsnorm_bf16(np.full((1, d), 0xBF00, np.uint16), g, 0.0)
    assert np.all(v == -1.0) and np.all(y == 0xBF80)


@pytest.mark.parametrize("k", [-40, -3, 5, 30])
def test_scale_invariance_without_epsilon(k):
    """eps = 0: scaling a row by 2^k changes no bit of v or y (each fp64 step scales exactly)."""
    x = _rows(31, 6, 300, lo=-8, hi=8)
    g = ig.rmsnorm_weight_bf16(32, 300)
    xs = ig.to_bf16_bits(ig.bf16_bits_to_f32(x).astype(np.float64) * 2.0**k)
    assert np.array_equal(ig.bf16_bits_to_f32(xs).astype(np.float64), ig.bf16_bits_to_f32(x) * 2.0**k)
    y1, v1 = oracle.rmsnorm_bf16(x, g, 0.0)
    y2, v2 = oracle.rmsnorm_bf16(xs, g, 0.0)
    assert np.array_equal(y1, y2) and np.array_equal(v1, v2)


def test_row_decomposition_and_row_selection():
    """RMSNorm([A; B]) = [RMSNorm(A); RMSNorm(B)] bitwise, and the rows= selection gives the
    same rows ("Batch-invariant RMSNorm": one row's reduction stays with that row)."""
    x = ig.scaled_rows_bf16(41, 20, 256)
    g = ig.rmsnorm_weight_bf16(42, 256)
    y, v = oracle.rmsnorm_bf16(x, g, 1e-6)
    for s in (1, 7, 19):
        ya, va = oracle.rmsnorm_bf16(x[:s], g, 1e-6)
        yb, vb = oracle.rmsnorm_bf16(x[s:], g, 1e-6)
        assert np.array_equal(np.vstack([ya, yb]), y) and np.array_equal(np.vstack([va, vb]), v)
    rows = [19, 0, 7, 7]
    ys, vs = oracle.rmsnorm_bf16(x, g, 1e-6, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(vs, v[rows])


def test_weight_applies_by_column():
    """A one-hot weight leaves one column; a ramp weight scales each column by its own g[j]
    (v[j] / (x[j] g[j]) is the same 1/rms for every j)."""
    d = 64
    x = ig.normal_bf16(51, 3, d)
    for j0 in (0, 5, d - 1):
        g = np.zeros(d, np.uint16)
        g[j0] = 0x3F80
        y, v = oracle.rmsnorm_bf16(x, g, 1e-6)
        nz = np.nonzero(v)[1]
        assert set(nz.tolist()) <= {j0} and np.all(v[:, j0] != 0)
    g = ig.to_bf16_bits(np.arange(1, d + 1, dtype=np.float64) / 8.0)
    _, v = oracle.rmsnorm_bf16(x, g, 1e-6)
    xf = ig.bf16_bits_to_f32(x).astype(np.float64)
    gf = ig.bf16_bits_to_f32(g).astype(np.float64)
    ratio = v / (xf * gf)
    assert np.all(np.abs(ratio - ratio[:, :1]) <= 4 * 2.0**-53 * np.abs(ratio[:, :1]))


def test_normalised_rows_have_unit_mean_square():
    x = ig.scaled_rows_bf16(61, 9, 4096)
    g = np.full(4096, 0x3F80, np.uint16)
    _, v = oracle.rmsnorm_bf16(x, g, 0.0)
    assert np.all(np.abs(np.mean(v * v, axis=1) - 1.0) <= 1e-13)


def test_against_torch_rms_norm_fp64():
    d = 4096
    x = ig.scaled_rows_bf16(71, 12, d)
    g = ig.rmsnorm_weight_bf16(72, d)
    eps = float(np.float32(1e-6))
    _, v = oracle.rmsnorm_bf16(x, g, eps)
    xt = torch.from_numpy(ig.bf16_bits_to_f32(x).astype(np.float64))
    gt = torch.from_numpy(ig.bf16_bits_to_f32(g).astype(np.float64))
    ref = torch.nn.functional.rms_norm(xt, (d,), gt, eps).numpy()
    assert np.all(np.abs(v - ref) <= 1e-14 * np.abs(ref) + 1e-300)


def _mutant(kind: str):
    """The oracle's definition with one plausible mistake, written out in numpy fp64."""
    def run(x, g, eps):
        xf = ig.bf16_bits_to_f32(x).astype(np.float64)
        gf = ig.bf16_bits_to_f32(g).astype(np.float64)
        d = x.shape[1]
        ss = np.sum(xf * xf, axis=1, keepdims=True)
        if kind == "mean_over_d_minus_1":
            ms = ss / (d - 1)
        else:
            ms = ss / d
        e = 0.0 if kind == "no_epsilon" else eps
        w = gf[::-1] if kind == "reversed_weight" else gf
        v = (xf * (1.0 / np.sqrt(ms + e))) * w
        return ig.to_bf16_bits(v), v
    return run


@pytest.mark.parametrize("kind", ["mean_over_d_minus_1", "no_epsilon", "reversed_weight"])
def test_planted_mistakes_fail_the_exact_check(kind):
    d, eps = 16, 0.0625
    x = _rows(81, 3, d, lo=-3, hi=0)
    g = ig.rmsnorm_weight_bf16(82, d)
    y, v = oracle.rmsnorm_bf16(x, g, eps)
    assert _agrees_exactly(y, v, x, g, eps)
    ym, vm = _mutant(kind)(x, g, eps)
    assert not _agrees_exactly(ym, vm, x, g, eps)


def test_tolerance_covers_fp32_arithmetic_then_bf16_rounding():
    """The GPU tolerance |y - v| <= (2^-8 + 2^-16)|v|: an fp32 evaluation with the sum of
    squares taken sequentially over the whole row (a worse order than any fixed tree), a
    correctly rounded reciprocal square root perturbed by 2 ulp, then bf16 rounding, stays
    inside it at d = 16384 for every element."""
    d = 16384
    x = ig.scaled_rows_bf16(91, 6, d)
    g = ig.rmsnorm_weight_bf16(92, d)
    eps = np.float32(1e-6)
    _, v = oracle.rmsnorm_bf16(x, g, float(eps))
    xf = ig.bf16_bits_to_f32(x)
    gf = ig.bf16_bits_to_f32(g)
    for i in range(x.shape[0]):
        ss = np.float32(0)
        for t in xf[i]:
            ss = np.float32(ss + np.float32(t * t))
        ms = np.float32(ss / np.float32(d))
        r = np.float32(1) / np.sqrt(np.float32(ms + eps))
        for ulps in (-2, 2):
            rr = np.float32(r * np.float32(1 + ulps * 2.0**-23))
            yv = ig.bf16_bits_to_f32(ig.to_bf16_bits((xf[i] * rr).astype(np.float32) * gf)).astype(np.float64)
            assert np.all(np.abs(yv - v[i]) <= oracle.TOL_RMSNORM_REL * np.abs(v[i]))


def test_bad_arguments_rejected():
    x = np.zeros((2, 8), np.uint16)
    g = np.zeros(8, np.uint16)
    with pytest.raises(ValueError):
        oracle.rmsnorm_bf16(x, g, -1.0)
    with pytest.raises(ValueError):
        oracle.rmsnorm_bf16(x, g, float("nan"))
    with pytest.raises(ValueError):
        oracle.rmsnorm_bf16(x, g, 0.0, rows=[2])
    with pytest.raises(ValueError):
        oracle.rmsnorm_bf16(np.zeros((2, 0), np.uint16), np.zeros(0, np.uint16), 0.0)


def test_exact_sqrt_rounding_helper():
    """The test-side square-root rounding: squares of bf16 values come back exactly, squared
    midpoints go to the even neighbour, and a hair above or below a midpoint decides it."""
    for b in (0x0081, 0x3F80, 0x3F81, 0x4049, 0x5A5A, 0x7F7D):
        v, up = bf16_value(b), bf16_value(b + 1)
        assert bf16_bits_of_signed_sqrt(v * v, False) == b
        assert bf16_bits_of_signed_sqrt(v * v, True) == 0x8000 | b
        m = (v + up) / 2
        even = b if b % 2 == 0 else b + 1
        assert bf16_bits_of_signed_sqrt(m * m, False) == even
        tiny = m * m * Fraction(1, 2**60)
        assert bf16_bits_of_signed_sqrt(m * m + tiny, False) == b + 1
        assert bf16_bits_of_signed_sqrt(m * m - tiny, False) == b
    assert bf16_bits_of_signed_sqrt(Fraction(0), True) == 0x8000
