"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes a loaded :class:`oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with:

- hand-derived closed forms (``tests/golden/closed_forms.txt``),
- an independent brute force (exact rationals + search among representable
  BF16 values, ``tests/bruteforce.py``) on tiny random inputs, including
  subnormals, huge exponents and cancellations,
- exact invariants of the definition (permuting k, permuting rows of W,
  scaling by powers of two, negation, independence of the rows of x, linearity
  of the exact sum, independence of the thread count),
- a float64 library matmul (agreement up to one BF16 ulp, nearly always exact).

The FP32-output form of the oracle has pins of its own (``pin_f32_*``): the
brute force's exact-integer FP32 rounding on tiny inputs, hand-derived ties,
overflow and subnormal cases, negation and power-of-two scaling, and a float64
library matmul converted to float32.

The same pins run against copies of the oracle with planted mistakes, which
must fail at least one of them (``test_oracle_pins.py``).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

import bruteforce
import golden_cases
from bf16_skinny_gemm_gb300 import synth
from tolerance import bits_to_f64


def _rng(seed):
    return np.random.default_rng(seed)


def wild_bits(rng, shape, exp_lo=100, exp_hi=154, p_zero=0.1, p_sub=0.05, p_huge=0.03):
    """Random finite BF16 bit patterns with a spread of exponents, some zeros,
    some subnormals and a few huge values."""
    n = int(np.prod(shape))
    sign = rng.integers(0, 2, n, dtype=np.uint16) << 15
    frac = rng.integers(0, 128, n, dtype=np.uint16)
    expo = rng.integers(exp_lo, exp_hi + 1, n).astype(np.uint16)
    u = rng.random(n)
    expo = np.where(u < p_sub, 0, expo)
    expo = np.where((u >= p_sub) & (u < p_sub + p_huge), rng.integers(200, 255, n), expo)
    b = (sign | (expo.astype(np.uint16) << 7) | frac).astype(np.uint16)
    b = np.where(rng.random(n) < p_zero, np.uint16(0), b)
    return b.reshape(shape).astype(np.uint16)


def _same(y, nan_mask, y_exp, nan_exp, what):
    assert np.array_equal(nan_mask, nan_exp), f"{what}: NaN pattern differs"
    sel = ~nan_exp
    if not np.array_equal(y[sel], y_exp[sel]):
        idx = np.argwhere((y != y_exp) & sel)[0]
        raise AssertionError(f"{what}: first mismatch at {tuple(idx)}: "
                             f"oracle {y[tuple(idx)]:#06x} expected {y_exp[tuple(idx)]:#06x}")


def _isnan_bits(y):
    return ((y & 0x7F80) == 0x7F80) & ((y & 0x007F) != 0)


def pin_golden(orc):
    for c in golden_cases.load():
        y = orc.skinny_gemm(c.x, c.W)
        _same(y, _isnan_bits(y), c.y, c.y_nan, f"golden case {c.name}")


def pin_bruteforce_wild(orc, seeds=range(12)):
    for s in seeds:
        rng = _rng(1000 + s)
        M = 1 + s % 4
        N = 1 + (3 * s) % 7
        K = [1, 2, 3, 7, 8, 16, 31, 48, 64, 5, 40, 24][s % 12]
        # alternate narrow exponent windows (heavy cancellation) and wide ones
        lo, hi = ((120, 134) if s % 2 else (60, 200))
        x = wild_bits(rng, (M, K), lo, hi)
        W = wild_bits(rng, (N, K), lo, hi)
        y = orc.skinny_gemm(x, W)
        yb, nb = bruteforce.gemm(x, W)
        _same(y, _isnan_bits(y), yb, nb, f"brute force (seed {s}, M{M} N{N} K{K})")


def pin_bruteforce_subnormal_region(orc, seeds=range(4)):
    """Products that land around the BF16 subnormal range (round to 2^-133 units)."""
    for s in seeds:
        rng = _rng(2000 + s)
        x = wild_bits(rng, (2, 12), 55, 72, p_sub=0.2, p_huge=0.0)
        W = wild_bits(rng, (5, 12), 55, 72, p_sub=0.2, p_huge=0.0)
        y = orc.skinny_gemm(x, W)
        yb, nb = bruteforce.gemm(x, W)
        _same(y, _isnan_bits(y), yb, nb, f"subnormal region (seed {s})")


def pin_bruteforce_gaussian(orc):
    x = synth.bits(synth.normal_bf16((4, 96), 1.0, seed=7))
    W = synth.bits(synth.normal_bf16((9, 96), 0.02, seed=8))
    y = orc.skinny_gemm(x, W)
    yb, nb = bruteforce.gemm(x, W)
    _same(y, _isnan_bits(y), yb, nb, "gaussian brute force")


def pin_exact_sum(orc):
    """The unrounded sum itself equals the exact rational sum."""
    rng = _rng(3)
    for K in (1, 3, 17, 64):
        x = wild_bits(rng, (K,), 40, 220)
        w = wild_bits(rng, (K,), 40, 220)
        v, bits = orc.exact_dot(x, w)
        ref = bruteforce.exact_dot(x, w)
        assert v == ref, f"exact sum differs at K={K}: {v} vs {ref}"
        assert bits == bruteforce.round_bf16(ref), f"rounding of exact sum differs at K={K}"
    # 2^100 + 1 - 2^100
    v, bits = orc.exact_dot(np.array([0x3F80] * 3, np.uint16),
                            np.array([0x7180, 0x3F80, 0xF180], np.uint16))
    assert v == 1 and bits == 0x3F80, "cancellation lost the small term"


def pin_large_constant(orc):
    for K, expect in ((256, 0x4380), (8192, 0x4600), (12288, 0x4640)):
        one = np.full((1, K), 0x3F80, np.uint16)
        y = orc.skinny_gemm(one, one)
        assert y[0, 0] == expect, f"sum of {K} ones gave {y[0, 0]:#06x}"
    # x = 1: y[n] is the correctly rounded row sum of W
    W = synth.bits(synth.normal_bf16((6, 512), 0.02, seed=11))
    y = orc.skinny_gemm(np.full((1, 512), 0x3F80, np.uint16), W)
    for n in range(6):
        s = sum((Fraction(bruteforce.bf16_to_float(b)) for b in W[n]), Fraction(0))
        assert y[0, n] == bruteforce.round_bf16(s), f"row sum {n}"


def pin_k_permutation(orc):
    rng = _rng(5)
    x = synth.bits(synth.normal_bf16((3, 2048), 1.0, seed=21))
    W = synth.bits(synth.normal_bf16((40, 2048), 0.02, seed=22))
    p = rng.permutation(2048)
    assert np.array_equal(orc.skinny_gemm(x, W), orc.skinny_gemm(x[:, p], W[:, p])), \
        "permuting k changed the result"


def pin_row_permutation(orc):
    rng = _rng(6)
    x = synth.bits(synth.normal_bf16((2, 300), 1.0, seed=23))
    W = synth.bits(synth.normal_bf16((33, 300), 0.02, seed=24))
    p = rng.permutation(33)
    assert np.array_equal(orc.skinny_gemm(x, W)[:, p], orc.skinny_gemm(x, W[p])), \
        "permuting rows of W did not permute y"


def pin_scaling(orc):
    x_t = synth.normal_bf16((2, 640), 1.0, seed=25)
    W = synth.bits(synth.normal_bf16((20, 640), 0.02, seed=26))
    for j in (-9, 5):
        xs = (x_t.double() * 2.0 ** j).to(torch.bfloat16)  # exact: power-of-two scale
        y1 = bits_to_f64(orc.skinny_gemm(synth.bits(x_t), W))
        y2 = bits_to_f64(orc.skinny_gemm(synth.bits(xs), W))
        assert np.array_equal(y2, y1 * 2.0 ** j), f"scaling x by 2^{j} did not scale y"


def pin_negation(orc):
    x = synth.bits(synth.normal_bf16((2, 500), 1.0, seed=27))
    W = synth.bits(synth.normal_bf16((25, 500), 0.02, seed=28))
    y1 = bits_to_f64(orc.skinny_gemm(x, W))
    y2 = bits_to_f64(orc.skinny_gemm(x ^ np.uint16(0x8000), W))
    assert np.array_equal(y2, -y1), "negating x did not negate y"


def pin_rows_independent(orc):
    x = synth.bits(synth.normal_bf16((4, 1000), 1.0, seed=29))
    W = synth.bits(synth.normal_bf16((17, 1000), 0.02, seed=30))
    y = orc.skinny_gemm(x, W)
    for m in range(4):
        assert np.array_equal(y[m:m + 1], orc.skinny_gemm(x[m:m + 1], W)), f"row {m}"


def pin_linearity(orc):
    """s(x1 + x2) = s(x1) + s(x2) exactly, for x1, x2 with disjoint support."""
    rng = _rng(9)
    K = 257
    w = wild_bits(rng, (K,), 90, 170)
    x1 = wild_bits(rng, (K,), 90, 170)
    mask = rng.random(K) < 0.5
    x2 = np.where(mask, x1, np.uint16(0)).astype(np.uint16)
    x1 = np.where(mask, np.uint16(0), x1).astype(np.uint16)
    x12 = (x1 | x2).astype(np.uint16)  # disjoint support: the sum is exact
    s1, _ = orc.exact_dot(x1, w)
    s2, _ = orc.exact_dot(x2, w)
    s12, _ = orc.exact_dot(x12, w)
    assert s12 == s1 + s2, "exact sums are not additive"
    s_dbl, _ = orc.exact_dot(x1, w)
    x1x2 = (synth.from_bits(x1).double() * 2).to(torch.bfloat16)
    s_two, _ = orc.exact_dot(synth.bits(x1x2), w)
    assert s_two == 2 * s_dbl, "s(2 x) != 2 s(x)"


def pin_threads(orc):
    x = synth.bits(synth.normal_bf16((3, 700), 1.0, seed=31))
    W = synth.bits(synth.normal_bf16((101, 700), 0.02, seed=32))
    assert np.array_equal(orc.skinny_gemm(x, W, threads=1), orc.skinny_gemm(x, W, threads=7)), \
        "thread count changed the result"


def pin_float64_library(orc):
    """A float64 library matmul, rounded to BF16, agrees within one ulp and is
    nearly always bitwise equal (float64 keeps ~45 more bits than BF16)."""
    xt = synth.normal_bf16((4, 1536), 1.0, seed=33)
    Wt = synth.normal_bf16((300, 1536), 0.02, seed=34)
    y = orc.skinny_gemm(synth.bits(xt), synth.bits(Wt))
    lib = (xt.double() @ Wt.double().T)
    lib_bits = synth.bits(lib.to(torch.bfloat16))
    frac_equal = float(np.mean(lib_bits == y))
    assert frac_equal >= 0.99, f"only {frac_equal:.4f} of outputs equal the float64 library's"
    d = np.abs(bits_to_f64(lib_bits) - bits_to_f64(y))
    from tolerance import ulp_bf16
    assert np.all(d <= ulp_bf16(bits_to_f64(y))), "float64 library differs by more than one ulp"


# ------------------------------------------------------------ FP32 outputs
def _f32_nan(y):
    return ((y & 0x7F800000) == 0x7F800000) & ((y & 0x007FFFFF) != 0)


def _f32_values(y):
    return np.asarray(y, np.uint32).view(np.float32).astype(np.float64)


def pin_f32_bruteforce_wild(orc, seeds=range(12)):
    """FP32 outputs against the brute force's exact-integer rounding, with
    cancellation, huge values (overflow to inf) and subnormal inputs."""
    for s in seeds:
        rng = _rng(5000 + s)
        M, N = 1 + s % 4, 1 + (5 * s) % 7
        K = [1, 2, 3, 8, 16, 31, 48, 64, 5, 40, 24, 7][s % 12]
        lo, hi = ((120, 134) if s % 2 else (60, 200))
        x = wild_bits(rng, (M, K), lo, hi)
        W = wild_bits(rng, (N, K), lo, hi)
        y = orc.skinny_gemm_f32(x, W)
        yb, nb = bruteforce.gemm_f32(x, W)
        _same(y, _f32_nan(y), yb, nb, f"FP32 brute force (seed {s}, M{M} N{N} K{K})")


def pin_f32_bruteforce_subnormal_region(orc, seeds=range(4)):
    """Products landing around the FP32 subnormal range (units of 2^-149)."""
    for s in seeds:
        rng = _rng(6000 + s)
        x = wild_bits(rng, (2, 10), 48, 66, p_sub=0.1, p_huge=0.0)
        W = wild_bits(rng, (4, 10), 48, 66, p_sub=0.1, p_huge=0.0)
        y = orc.skinny_gemm_f32(x, W)
        yb, nb = bruteforce.gemm_f32(x, W)
        _same(y, _f32_nan(y), yb, nb, f"FP32 subnormal region (seed {s})")


def pin_f32_closed_forms(orc):
    """Hand-derived FP32 results (BF16 bits: 1 = 0x3F80, 2^-24 = 0x3380, 2^-30 =
    0x3080, 1 + 2^-7 = 0x3F81, 2^127 = 0x7F00, 4 = 0x4080, 2 - 2^-7 = 0x3FFF,
    2^-75 = 0x1A00, 1.5 * 2^-75 = 0x1A40)."""
    cases = [
        # 1 + 2^-24: exactly half an FP32 ulp above 1, ties to the even 1.0
        ([0x3F80, 0x3F80], [0x3F80, 0x3380], 0x3F800000),
        # 1 + 2^-24 + 2^-30: above the midpoint, rounds up to 1 + 2^-23
        ([0x3F80] * 3, [0x3F80, 0x3380, 0x3080], 0x3F800001),
        # (1 + 2^-7) + 2^-24: a tie again; 0x3F810000 has an even significand, so it stays
        ([0x3F80, 0x3F80], [0x3F81, 0x3380], 0x3F810000),
        # 2^127 * 4 = 2^129 overflows to +inf
        ([0x7F00], [0x4080], 0x7F800000),
        # 2^127 * (2 - 2^-7) = 2^128 - 2^120: 8 significand bits, exact, finite
        ([0x7F00], [0x3FFF], 0x7F7F0000),
        # 2^-150: half the smallest subnormal 2^-149, ties to the even +0
        ([0x1A00], [0x1A00], 0x00000000),
        # 1.5 * 2^-150 = 0.75 * 2^-149: rounds to the smallest subnormal
        ([0x1A00], [0x1A40], 0x00000001),
        # -(1 + 2^-24 + 2^-30): the sign does not change the magnitude's rounding
        ([0xBF80] * 3, [0x3F80, 0x3380, 0x3080], 0xBF800001),
    ]
    for xs, ws, expect in cases:
        y = orc.skinny_gemm_f32(np.array([xs], np.uint16), np.array([ws], np.uint16))
        assert y[0, 0] == expect, f"FP32 closed form {xs}.{ws}: {y[0, 0]:#010x} != {expect:#010x}"
    # 12289 ones: exact in FP32 (BF16 would give 12288); encoded by the host's float32
    one = np.full((1, 12289), 0x3F80, np.uint16)
    expect = int(np.array([12289.0], np.float32).view(np.uint32)[0])
    assert orc.skinny_gemm_f32(one, one)[0, 0] == expect, "sum of 12289 ones"


def pin_f32_negation_and_scaling(orc):
    x_t = synth.normal_bf16((2, 640), 1.0, seed=41)
    W = synth.bits(synth.normal_bf16((20, 640), 0.02, seed=42))
    y1 = _f32_values(orc.skinny_gemm_f32(synth.bits(x_t), W))
    y_neg = _f32_values(orc.skinny_gemm_f32(synth.bits(x_t) ^ np.uint16(0x8000), W))
    assert np.array_equal(y_neg, -y1), "negating x did not negate the FP32 outputs"
    for j in (-9, 5):
        xs = (x_t.double() * 2.0 ** j).to(torch.bfloat16)
        y2 = _f32_values(orc.skinny_gemm_f32(synth.bits(xs), W))
        assert np.array_equal(y2, y1 * 2.0 ** j), f"scaling x by 2^{j} did not scale y"


def pin_f32_float64_library(orc):
    """A float64 library matmul converted to float32 agrees within one FP32 ulp
    and nearly always bitwise (float64 keeps 29 more bits than FP32)."""
    xt = synth.normal_bf16((4, 4096), 1.0, seed=43)
    Wt = synth.normal_bf16((288, 4096), 0.02, seed=44)
    y = orc.skinny_gemm_f32(synth.bits(xt), synth.bits(Wt))
    lib = (xt.double() @ Wt.double().T).numpy().astype(np.float32).view(np.uint32)
    frac_equal = float(np.mean(lib == y))
    assert frac_equal >= 0.999, f"only {frac_equal:.4f} of FP32 outputs equal the library's"
    d = np.abs(lib.astype(np.int64) - y.astype(np.int64))   # same sign here: ulps apart
    assert np.all(d <= 1), "float64 library differs by more than one FP32 ulp"


ALL_PINS = [pin_golden, pin_bruteforce_wild, pin_bruteforce_subnormal_region,
            pin_bruteforce_gaussian, pin_exact_sum, pin_large_constant, pin_k_permutation,
            pin_row_permutation, pin_scaling, pin_negation, pin_rows_independent,
            pin_linearity, pin_threads, pin_float64_library,
            pin_f32_bruteforce_wild, pin_f32_bruteforce_subnormal_region, pin_f32_closed_forms,
            pin_f32_negation_and_scaling, pin_f32_float64_library]
