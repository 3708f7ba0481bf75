"""Exact rational restatement of the quantiser's per-element arithmetic, for pins.

Written from the formats' definitions with Python fractions, independently of
the oracle: IEEE binary32 round-to-nearest-even (subnormals included) and the
OCP E4M3FN grid (bias 7, 3 fraction bits, largest finite 448) with
round-to-nearest-even and saturation. The quantiser's definition (one FP32
scale s = amax / 448 per tile, code = e4m3(fl32(x / s)), as the Puro-2B
recipe's DeepSeek-V3-style blockwise FP8 is read) composes these steps.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def _floor_log2(a: Fraction) -> int:
    """e with 2^e <= a < 2^(e+1), for a > 0."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def _round_half_even(q: Fraction) -> int:
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def rn32(q: Fraction) -> Fraction:
    """The binary32 value nearest to q (ties to even), subnormals included; q finite, in range."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = max(_floor_log2(a), -126)
    ulp = Fraction(2) ** (e - 23)
    return sign * _round_half_even(a / ulp) * ulp


def f32(v: float) -> Fraction:
    """Exact value of a binary32 number."""
    return Fraction(float(np.float32(v)))


def bf16_value(bits: int) -> Fraction:
    """Exact value of a bfloat16 bit pattern (finite)."""
    return Fraction(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))


def e4m3_code(t: Fraction, negative_zero: bool = False) -> int:
    """E4M3FN code of t: nearest grid value (ties to even), magnitudes above 448 saturate to 448."""
    sign = 0x80 if (t < 0 or (t == 0 and negative_zero)) else 0x00
    a = abs(t)
    if a == 0:
        return sign
    e = _floor_log2(a)
    spacing = Fraction(2) ** (-9) if e < -6 else Fraction(2) ** (e - 3)
    v = _round_half_even(a / spacing) * spacing
    if v > 448:
        v = Fraction(448)
    if v == 0:
        return sign
    if v < Fraction(2) ** -6:
        return sign | int(v / Fraction(2) ** -9)
    e2 = _floor_log2(v)
    m = int(v / Fraction(2) ** e2 * 8) - 8
    return sign | ((e2 + 7) << 3) | m


def tile_scale(amax: Fraction) -> Fraction:
    """s = fl32(amax / 448)."""
    return rn32(amax / 448)


def code_by_definition(amax: Fraction, x: Fraction, x_negative_zero: bool = False) -> int:
    """code = e4m3(fl32(x / s)), s = fl32(amax / 448); an all-zero tile (s = 0) gives signed zeros."""
    s = tile_scale(amax)
    if s == 0:
        return 0x80 if (x < 0 or x_negative_zero) else 0x00
    return e4m3_code(rn32(x / s), x_negative_zero)


def code_by_reciprocal(amax: Fraction, x: Fraction) -> int:
    """The rejected reading e4m3(fl32(x * fl32(1 / s))): one rounding more than the definition."""
    s = tile_scale(amax)
    return e4m3_code(rn32(x * rn32(1 / s)))


def code_by_single_rounding(amax: Fraction, x: Fraction) -> int:
    """The rejected reading e4m3(x / s): the exact quotient rounded once, straight to E4M3."""
    s = tile_scale(amax)
    return e4m3_code(x / s)
