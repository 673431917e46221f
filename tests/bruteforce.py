"""Brute-force reference for tiny inputs, independent of the oracle's code.

It shares nothing with ``oracle/skinny_oracle.c``:

- BF16 bits are decoded by the host's float32 hardware (``struct``), then
  turned into exact ``Fraction`` values;
- the dot product is summed in exact rational arithmetic;
- rounding to BF16 does not manipulate bits: it searches the sorted list of all
  finite BF16 values for the two neighbours of the exact value and picks the
  nearer one, the one with an even significand on a tie, and +-inf at or
  beyond the midpoint between the largest finite value and 2^128 (IEEE 754
  roundTiesToEven with overflow).
"""
from __future__ import annotations

import bisect
import math
import struct
from fractions import Fraction

import numpy as np


def bf16_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]


# finite non-negative BF16 values in bit order 0x0000..0x7f7f (monotone increasing)
_POS_VALUES = [bf16_to_float(b) for b in range(0x0000, 0x7F80)]
_MAX_FINITE = Fraction(_POS_VALUES[-1])
_OVERFLOW_MIDPOINT = (_MAX_FINITE + Fraction(2) ** 128) / 2


def round_bf16(v: Fraction) -> int:
    """BF16 bits of the exact rational ``v`` under roundTiesToEven."""
    if v == 0:
        return 0x0000
    sign = 0x8000 if v < 0 else 0x0000
    a = abs(v)
    if a >= _OVERFLOW_MIDPOINT:
        return sign | 0x7F80
    i = bisect.bisect_left(_POS_VALUES, a)   # _POS_VALUES[i-1] < a <= _POS_VALUES[i]
    if i < len(_POS_VALUES) and Fraction(_POS_VALUES[i]) == a:
        return sign | i
    lo, hi = i - 1, i
    if hi == len(_POS_VALUES):               # between max finite and the midpoint
        return sign | lo
    d_lo = a - Fraction(_POS_VALUES[lo])
    d_hi = Fraction(_POS_VALUES[hi]) - a
    if d_lo < d_hi:
        return sign | lo
    if d_hi < d_lo:
        return sign | hi
    return sign | (lo if lo % 2 == 0 else hi)


_F32_MAX = (Fraction(2) ** 24 - 1) * Fraction(2) ** 104


def round_f32(v: Fraction) -> int:
    """FP32 bits of the exact rational ``v`` under roundTiesToEven, by exact
    integer arithmetic: find the binade, scale so the ulp is 1, round the
    quotient half to even, carry into the next binade, and overflow to +-inf
    at or beyond the midpoint between the largest finite value and 2^128."""
    if v == 0:
        return 0x00000000
    sign = 0x80000000 if v < 0 else 0
    a = abs(v)
    if a >= (_F32_MAX + Fraction(2) ** 128) / 2:
        return sign | 0x7F800000
    e = a.numerator.bit_length() - a.denominator.bit_length()   # 2^e <= a < 2^(e+2)
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    u = max(e - 23, -149)                      # exponent of the ulp
    q = a / Fraction(2) ** u
    qi = q.numerator // q.denominator
    rem = q - qi
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and qi % 2 == 1):
        qi += 1
    if qi == 1 << 24:                           # carried into the next binade
        qi, u = 1 << 23, u + 1
    if u > 104:
        return sign | 0x7F800000
    if qi < (1 << 23):                          # subnormal
        return sign | qi
    return sign | ((u + 150) << 23) | (qi - (1 << 23))


def exact_dot(x_row, w_row):
    """Exact sum of products: a Fraction, or 'nan' / '+inf' / '-inf'."""
    xs = [bf16_to_float(b) for b in x_row]
    ws = [bf16_to_float(b) for b in w_row]
    if any(not math.isfinite(v) for v in xs + ws):
        # products of finite BF16 values never overflow a double, so IEEE double
        # arithmetic gives the right special value here
        s = sum(a * b for a, b in zip(xs, ws))
        if math.isnan(s):
            return "nan"
        return "+inf" if s > 0 else "-inf"
    return sum((Fraction(a) * Fraction(b) for a, b in zip(xs, ws)), Fraction(0))


def gemm_f32(x_bits: np.ndarray, W_bits: np.ndarray):
    """(y FP32 bits [M,N] as uint32, nan mask [M,N]) for tiny inputs."""
    M, N = x_bits.shape[0], W_bits.shape[0]
    y = np.zeros((M, N), dtype=np.uint32)
    nan = np.zeros((M, N), dtype=bool)
    for m in range(M):
        for n in range(N):
            s = exact_dot(x_bits[m], W_bits[n])
            if s == "nan":
                nan[m, n] = True
            elif s == "+inf":
                y[m, n] = 0x7F800000
            elif s == "-inf":
                y[m, n] = 0xFF800000
            else:
                y[m, n] = round_f32(s)
    return y, nan


def gemm(x_bits: np.ndarray, W_bits: np.ndarray):
    """(y bits [M,N], nan mask [M,N]) for tiny inputs."""
    M, N = x_bits.shape[0], W_bits.shape[0]
    y = np.zeros((M, N), dtype=np.uint16)
    nan = np.zeros((M, N), dtype=bool)
    for m in range(M):
        for n in range(N):
            s = exact_dot(x_bits[m], W_bits[n])
            if s == "nan":
                nan[m, n] = True
            elif s == "+inf":
                y[m, n] = 0x7F80
            elif s == "-inf":
                y[m, n] = 0xFF80
            else:
                y[m, n] = round_bf16(s)
    return y, nan
