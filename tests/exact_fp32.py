"""Exact rational arithmetic used to pin binary32 results independently of any C library.

fma_f32(a, b, c) is the definition of a fused multiply-add: the exact value a*b + c rounded
once to the nearest binary32 (ties to even). Nothing here calls the oracle or the GPU code.
"""
from __future__ import annotations

import struct
from fractions import Fraction

import numpy as np

_F32_MAX = Fraction(2) ** 127 * (2 - Fraction(1, 2**23))


def bits(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(np.float32(x))))[0]


def from_bits(b: int) -> np.float32:
    return np.frombuffer(struct.pack("<I", b & 0xFFFFFFFF), dtype=np.float32)[0]


def key(x) -> int:
    return bits(x) & 0x7FFFFFFF


def round_f32(q: Fraction) -> np.float32:
    """Round an exact rational to binary32, nearest with ties to even (finite inputs)."""
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum_exp = max(e, -126) - 23
    scaled = a / Fraction(2) ** quantum_exp
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    val = m * Fraction(2) ** quantum_exp
    if val > _F32_MAX:
        return np.float32(sign * np.inf)
    return np.float32(sign * float(val))


def _zero_sum_sign(neg_p: bool, neg_c: bool, p_zero: bool, c_zero: bool) -> np.float32:
    # IEEE 754, round to nearest: an exact zero sum is -0 only when both addends are -0.
    if p_zero and c_zero and neg_p and neg_c:
        return np.float32(-0.0)
    return np.float32(0.0)


def fma_f32(a, b, c) -> np.float32:
    a, b, c = np.float32(a), np.float32(b), np.float32(c)
    q = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    if q == 0:
        return _zero_sum_sign(bool(np.signbit(a)) != bool(np.signbit(b)), bool(np.signbit(c)),
                              a == 0 or b == 0, c == 0)
    return round_f32(q)


def add_f32(a, b) -> np.float32:
    a, b = np.float32(a), np.float32(b)
    q = Fraction(float(a)) + Fraction(float(b))
    if q == 0:
        return _zero_sum_sign(bool(np.signbit(a)), bool(np.signbit(b)), a == 0, b == 0)
    return round_f32(q)


def mul_f32(a, b) -> np.float32:
    a, b = np.float32(a), np.float32(b)
    q = Fraction(float(a)) * Fraction(float(b))
    if q == 0:
        return np.float32(-0.0) if bool(np.signbit(a)) != bool(np.signbit(b)) else np.float32(0.0)
    return round_f32(q)
