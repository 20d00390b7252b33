"""Exact rational model of binary32 / bfloat16 arithmetic, for pinning the oracle.

This is an independent, deliberately slow statement of IEEE 754 rounding from
its textbook definition: a value is an exact ``fractions.Fraction`` (plus
signed zero and infinities), and rounding picks the nearest member of the
format's grid at the value's binade, ties to the even significand, with
overflow to infinity.  It uses no bit manipulation and none of the oracle's
code, so an error in the oracle's bit-level rounding or in its order of
additions shows up as a disagreement.
"""

from __future__ import annotations

import math
import struct
from fractions import Fraction

INF = "inf"
NINF = "-inf"
NAN = "nan"

# (precision incl. the implicit bit, minimum normal exponent, maximum exponent)
BINARY32 = (24, -126, 127)
BFLOAT16 = (8, -126, 127)


class Val:
    """An IEEE value: finite Fraction with a sign for zero, or inf / -inf / nan."""

    __slots__ = ("kind", "q", "neg")

    def __init__(self, kind: str, q: Fraction = Fraction(0), neg: bool = False):
        self.kind, self.q, self.neg = kind, q, neg

    @staticmethod
    def finite(q: Fraction, neg_zero: bool = False) -> "Val":
        return Val("fin", q, neg_zero if q == 0 else q < 0)

    def __repr__(self):  # pragma: no cover
        return f"Val({self.kind}, {self.q}, neg={self.neg})"


def _floor_log2(q: Fraction) -> int:
    """floor(log2(q)) for a positive Fraction, exactly."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    return e


def round_to(v: Val, fmt) -> Val:
    """Round to the nearest value of the format, ties to even significand."""
    if v.kind != "fin" or v.q == 0:
        return v
    p, emin, emax = fmt
    mag = abs(v.q)
    e = max(_floor_log2(mag), emin)
    ulp = Fraction(2) ** (e - p + 1)
    scaled = mag / ulp
    m = math.floor(scaled)
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    r = m * ulp
    if r >= Fraction(2) ** (emax + 1):
        return Val(NINF if v.q < 0 else INF)
    if r == 0:
        return Val("fin", Fraction(0), v.q < 0)
    return Val("fin", r if v.q > 0 else -r, v.q < 0)


def add(a: Val, b: Val) -> Val:
    """Exact sum before rounding, with IEEE's special-value and signed-zero rules."""
    if a.kind == NAN or b.kind == NAN:
        return Val(NAN)
    if a.kind in (INF, NINF) or b.kind in (INF, NINF):
        kinds = {a.kind, b.kind} - {"fin"}
        if kinds == {INF, NINF}:
            return Val(NAN)
        return Val(kinds.pop())
    s = a.q + b.q
    if s == 0:
        # Round to nearest: an exact zero sum is +0 unless both operands are -0.
        both_neg_zero = a.q == 0 and b.q == 0 and a.neg and b.neg
        return Val("fin", Fraction(0), both_neg_zero)
    return Val("fin", s, s < 0)


def from_bf16_bits(b: int) -> Val:
    u = (b & 0xFFFF) << 16
    f = struct.unpack("<f", struct.pack("<I", u))[0]
    if math.isnan(f):
        return Val(NAN)
    if math.isinf(f):
        return Val(INF if f > 0 else NINF)
    return Val("fin", Fraction(f), bool(b & 0x8000))


def to_bf16_bits(v: Val) -> int | None:
    """bf16 pattern of a value already on the bf16 grid (None for NaN)."""
    if v.kind == NAN:
        return None
    if v.kind == INF:
        return 0x7F80
    if v.kind == NINF:
        return 0xFF80
    if v.q == 0:
        return 0x8000 if v.neg else 0x0000
    f = float(v.q)  # exact: bf16 grid values are binary64 values
    u = struct.unpack("<I", struct.pack("<f", f))[0]
    assert u & 0xFFFF == 0, "value is not on the bf16 grid"
    return u >> 16


def rank_order_sum_bits(values: list[int]) -> int | None:
    """bf16 result of the rank-order fp32 sum of bf16 patterns (None = NaN)."""
    acc = Val("fin", Fraction(0), False)
    for b in values:
        acc = round_to(add(acc, from_bf16_bits(b)), BINARY32)
    return to_bf16_bits(round_to(acc, BFLOAT16))
