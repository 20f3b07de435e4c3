"""Exact-rational emulation of binary32 arithmetic, written from IEEE 754.

Independent of the C oracle and of the CUDA library: values are decoded from
their bit patterns into ``fractions.Fraction``, each operation is carried out
exactly, then rounded to the binary32 grid (24-bit significand, gradual
underflow below 2**-126, round to nearest with ties to even, overflow to
infinity) and finally flushed if the rounded result is subnormal.  Operands
that are subnormal are replaced by a zero of the same sign first.

This is the arithmetic model the pages' reproducible-ops rules ask for (a
rounded multiply and a rounded add, never fused; subnormals flushed on every
backend) and is used only to pin the oracle.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

P = 24          # significand bits
EMIN = -126     # smallest normal exponent
EMAX = 127
FLT_MIN = Fraction(1, 2 ** 126)
BIG = Fraction(2 ** 128)


class F32:
    """A binary32 value: sign bit, and either a finite magnitude or inf/nan."""

    __slots__ = ("neg", "mag", "kind")

    def __init__(self, neg: bool, mag: Fraction | None, kind: str = "fin"):
        self.neg = bool(neg)
        self.mag = mag
        self.kind = kind

    # -------- encoding
    @staticmethod
    def from_bits(b: int) -> "F32":
        b &= 0xFFFFFFFF
        neg = bool(b >> 31)
        e = (b >> 23) & 0xFF
        f = b & 0x7FFFFF
        if e == 0xFF:
            return F32(neg, None, "nan" if f else "inf")
        if e == 0:
            return F32(neg, Fraction(f, 2 ** 149))
        return F32(neg, Fraction(0x800000 | f) * Fraction(2) ** (e - 150))

    @staticmethod
    def from_float(x: float) -> "F32":
        return F32.from_bits(struct.unpack("<I", struct.pack("<f", x))[0])

    def bits(self) -> int:
        s = 0x80000000 if self.neg else 0
        if self.kind == "nan":
            return 0x7FC00000
        if self.kind == "inf":
            return s | 0x7F800000
        m = self.mag
        if m == 0:
            return s
        e = _floor_log2(m)
        if e < EMIN:  # subnormal
            f = m * 2 ** 149
            assert f.denominator == 1
            return s | int(f)
        f = m / Fraction(2) ** (e - 23)
        assert f.denominator == 1 and 0x800000 <= f < 0x1000000
        return s | ((e + 127) << 23) | (int(f) & 0x7FFFFF)

    def to_float(self) -> float:
        return struct.unpack("<f", struct.pack("<I", self.bits()))[0]

    def value(self) -> Fraction:
        assert self.kind == "fin"
        return -self.mag if self.neg else self.mag

    def is_zero(self) -> bool:
        return self.kind == "fin" and self.mag == 0

    def __repr__(self) -> str:
        return f"F32({self.to_float()!r}, bits=0x{self.bits():08x})"


def _floor_log2(m: Fraction) -> int:
    """Exact floor(log2(m)) for m > 0."""
    e = m.numerator.bit_length() - m.denominator.bit_length()
    if Fraction(2) ** e > m:
        e -= 1
    elif Fraction(2) ** (e + 1) <= m:
        e += 1
    return e


def _rne_int(x: Fraction) -> int:
    """Round a non-negative rational to the nearest integer, ties to even."""
    n = x.numerator // x.denominator
    r = x - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def round_to_f32(neg: bool, mag: Fraction) -> F32:
    """IEEE binary32 round-to-nearest-even of a signed exact magnitude
    (gradual underflow, overflow to infinity).  No flushing here."""
    if mag == 0:
        return F32(neg, Fraction(0))
    e = _floor_log2(mag)
    q = max(e, EMIN) - (P - 1)              # exponent of the quantum
    n = _rne_int(mag / Fraction(2) ** q)
    r = Fraction(n) * Fraction(2) ** q
    if r >= BIG:
        return F32(neg, None, "inf")
    return F32(neg, r)


def flush(x: F32) -> F32:
    """Subnormal -> zero of the same sign."""
    if x.kind == "fin" and 0 < x.mag < FLT_MIN:
        return F32(x.neg, Fraction(0))
    return x


def add(a: F32, b: F32) -> F32:
    a, b = flush(a), flush(b)
    assert a.kind == "fin" and b.kind == "fin"
    s = a.value() + b.value()
    if s == 0:
        # exact zero sum: -0 only when both addends are -0 (round to nearest)
        neg = a.is_zero() and b.is_zero() and a.neg and b.neg
        return F32(neg, Fraction(0))
    return flush(round_to_f32(s < 0, abs(s)))


def mul(a: F32, b: F32) -> F32:
    a, b = flush(a), flush(b)
    assert a.kind == "fin" and b.kind == "fin"
    return flush(round_to_f32(a.neg != b.neg, a.mag * b.mag))


def div(a: F32, b: F32) -> F32:
    a, b = flush(a), flush(b)
    neg = a.neg != b.neg
    # IEEE 754 special operands: NaN propagates; inf/inf and 0/0 are invalid
    # (NaN); inf/finite is inf; finite/inf is a signed zero; x/0 is inf
    if a.kind == "nan" or b.kind == "nan":
        return F32(False, None, "nan")
    if a.kind == "inf":
        return F32(False, None, "nan") if b.kind == "inf" else F32(neg, None, "inf")
    if b.kind == "inf":
        return F32(neg, Fraction(0))
    if b.is_zero():
        return F32(False, None, "nan") if a.is_zero() else F32(neg, None, "inf")
    return flush(round_to_f32(neg, a.mag / b.mag))


def sqrt(a: F32) -> F32:
    a = flush(a)
    assert a.kind == "fin"
    if a.is_zero():
        return F32(a.neg, Fraction(0))
    assert not a.neg
    m = a.mag
    e = _floor_log2(m)
    er = e // 2                      # floor(e/2): exponent of the root
    q = er - (P - 1)
    # x = m / 2^(2q); result significand n = RN(sqrt(x))
    x = m / Fraction(2) ** (2 * q)
    n = math.isqrt(x.numerator // x.denominator)
    # n = floor(sqrt(x)); decide between n and n+1 by the midpoint
    mid = Fraction(2 * n + 1, 2) ** 2
    if x > mid or (x == mid and n % 2 == 1):
        n += 1
    return flush(round_to_f32(False, Fraction(n) * Fraction(2) ** q))


def i2f(v: int) -> F32:
    return round_to_f32(v < 0, Fraction(abs(v)))


def rint_half_even(a: F32) -> int:
    """Nearest integer, ties to even (exact on the decoded value)."""
    v = a.value()
    n = _rne_int(abs(v))
    return -n if v < 0 else n


def quant(x: F32, s: F32, qmax: int = 127) -> int:
    s = flush(s)
    if s.is_zero():
        return 0
    v = div(x, s)
    if v.kind == "nan":
        return 0
    if v.kind == "inf":
        return -qmax if v.neg else qmax
    q = rint_half_even(v)
    return max(-qmax, min(qmax, q))


def f(x: float) -> F32:
    return F32.from_float(x)
