"""Exact rational arithmetic used to pin the oracle (test side only).

Everything here is written from the IEEE-754 / OCP format definitions with
Python's Fraction, independently of the oracle's C bit manipulation, so that a
mistake in either shows up as a disagreement.
"""
from __future__ import annotations

from fractions import Fraction


def bf16_value(bits: int) -> Fraction:
    """Exact value of a finite bf16 pattern: 1 sign, 8 exponent (bias 127), 7 mantissa bits."""
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    assert e != 0xFF, "not finite"
    if e == 0:
        return s * Fraction(m, 1) * Fraction(1, 2**133)          # m/128 * 2^-126
    return s * Fraction(128 + m) * _pow2(e - 134)


def f32_value(bits: int) -> Fraction:
    s = -1 if bits & 0x80000000 else 1
    e = (bits >> 23) & 0xFF
    m = bits & 0x7FFFFF
    assert e != 0xFF
    if e == 0:
        return s * Fraction(m) * _pow2(-149)
    return s * Fraction(2**23 + m) * _pow2(e - 150)


def e4m3_value(code: int) -> Fraction:
    """OCP E4M3FN: bias 7, subnormal m * 2^-9, S.1111.111 is NaN (not handled here)."""
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 7
    assert not (e == 0xF and m == 7)
    if e == 0:
        return s * Fraction(m) * _pow2(-9)
    return s * Fraction(8 + m) * _pow2(e - 10)


def e8m0_value(e: int) -> Fraction:
    assert e != 0xFF
    return _pow2(e - 127)


def _pow2(n: int) -> Fraction:
    return Fraction(2**n) if n >= 0 else Fraction(1, 2 ** (-n))


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while _pow2(e) > a:
        e -= 1
    while _pow2(e + 1) <= a:
        e += 1
    return e


def _rne_int(q: Fraction) -> int:
    """Round a non-negative rational to the nearest integer, ties to even."""
    f = q.numerator // q.denominator
    r = q - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def round_to_binary(v: Fraction, p: int, emin: int, emax: int):
    """Round v to the binary format with p significand bits (incl. hidden), exponent range
    [emin, emax]; returns (sign, units, qe) with value = sign * units * 2^qe, or None for
    overflow (the rounded magnitude exceeds the largest finite number)."""
    if v == 0:
        return (1, 0, emin - p + 1)
    sign = -1 if v < 0 else 1
    a = abs(v)
    lg = _floor_log2(a)
    qe = max(lg, emin) - (p - 1)
    units = _rne_int(a / _pow2(qe))
    if units == 2**p:
        units //= 2
        qe += 1
    if qe + (p - 1) > emax:
        return None
    return (sign, units, qe)


def to_bf16_bits_exact(v: Fraction) -> int:
    r = round_to_binary(v, 8, -126, 127)
    if r is None:
        return 0xFF80 if v < 0 else 0x7F80
    sign, units, qe = r
    sb = 0x8000 if sign < 0 else 0
    if units == 0:
        return sb
    if units < 128:                      # subnormal
        assert qe == -133
        return sb | units
    E = qe + 134
    return sb | (E << 7) | (units - 128)


def to_f32_bits_exact(v: Fraction) -> int:
    r = round_to_binary(v, 24, -126, 127)
    if r is None:
        return 0xFF800000 if v < 0 else 0x7F800000
    sign, units, qe = r
    sb = 0x80000000 if sign < 0 else 0
    if units == 0:
        return sb
    if units < 2**23:
        assert qe == -149
        return sb | units
    E = qe + 150
    return sb | (E << 23) | (units - 2**23)


def gamma(n: int, u: float) -> float:
    """gamma_n = n u / (1 - n u) ("Quantifying with unit roundoff", nondeterminism article)."""
    nu = n * u
    assert nu < 1
    return nu / (1 - nu)


def bf16_bits_of_signed_sqrt(q: Fraction, negative: bool) -> int:
    """Bits of RNE_bf16(+-sqrt(q)) for a rational q >= 0, decided exactly: the result r is the
    bf16 value whose rounding interval [mid(r-, r), mid(r, r+)] holds sqrt(q), tested by
    comparing q with the squared midpoints (ties go to the even pattern).  Finite normal
    results only (the tests keep their values inside the bf16 normal range)."""
    assert q >= 0
    sb = 0x8000 if negative else 0
    if q == 0:
        return sb
    b = to_bf16_bits_exact(Fraction(float(q) ** 0.5)) & 0x7FFF    # first guess, then fix up
    assert 0x0080 <= b < 0x7F80
    while True:
        v = bf16_value(b)
        lo = (bf16_value(b - 1) + v) / 2
        hi = (v + bf16_value(b + 1)) / 2
        if q < lo * lo or (q == lo * lo and b % 2 == 1):
            b -= 1
        elif q > hi * hi or (q == hi * hi and b % 2 == 1):
            b += 1
        else:
            return sb | b


def f32_bits_of_signed_sqrt(q: Fraction, negative: bool) -> int:
    """Bits of RNE_fp32(+-sqrt(q)) for a rational q >= 0, decided exactly as for bf16 above (the
    fp32 value whose rounding interval holds sqrt(q), by comparing q with squared midpoints).
    Finite normal results only."""
    assert q >= 0
    sb = 0x80000000 if negative else 0
    if q == 0:
        return sb
    b = to_f32_bits_exact(Fraction(float(q) ** 0.5)) & 0x7FFFFFFF
    assert 0x00800000 <= b < 0x7F800000
    while True:
        v = f32_value(b)
        lo = (f32_value(b - 1) + v) / 2
        hi = (v + f32_value(b + 1)) / 2
        if q < lo * lo or (q == lo * lo and b % 2 == 1):
            b -= 1
        elif q > hi * hi or (q == hi * hi and b % 2 == 1):
            b += 1
        else:
            return sb | b
