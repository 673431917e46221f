"""Acceptance checks for a GPU result against the oracle.

Two per-element bounds and one per-row cosine, all evaluated in float64:

1. The stated tolerance of the method (per element):
       |y_gpu - y_ref| <= 2 * ulp_bf16(|y_ref|) + 1e-3 * sqrt(K) * max|x| * max|W|
   with max|x| and max|W| taken over the whole call (per pair in a batched
   call).  ulp_bf16(v) = 2^(floor(log2 v) - 7) for a normal v and 2^-133 for
   zero or a subnormal.

2. A tighter bound derived from the arithmetic (per element).  Every product
   of two BF16 values is exact in FP32 (8-bit x 8-bit significands), so an FP32
   accumulation of K products in ANY order and grouping (sequential, tree,
   split-K partials summed later) differs from the exact sum s by at most
       e = gamma_(K-1) * sum_k |x_k W_k| + K * 2^-150,
   gamma_n = n u / (1 - n u), u = 2^-24 (the second term covers products that
   underflow FP32).  Rounding s and the FP32 sum to BF16 adds at most one ulp
   of the larger magnitude each side, hence
       |y_gpu - y_ref| <= 2 * ulp_bf16(|y_ref| + e) + e.

3. Cosine similarity of each output row y[m, :] with the oracle's, >= 0.99999
   (two all-zero rows count as equal).  The pages check cosine against
   F.linear (vLLM PR #62949, Validation); vLLM PR #65306 (Validation) uses a
   per-element float64 bound 7.5e-5 + 2^-8 |ref|, which is reported, not
   asserted, because it assumes unit-scale inputs.

Non-finite references must be matched in kind (NaN by NaN, +-inf by the same
infinity).

FP32 outputs (``compare_f32``): the GPU's FP32 sum differs from the exact sum by
at most e (bound 2), and the oracle's reference is the exact sum rounded once
to FP32, so |y_gpu - y_ref| <= e + ulp_f32(|y_ref|) / 2; the cosine check is the
same.  The spec element bound is stated for BF16 outputs and does not
apply.
"""
from __future__ import annotations

import numpy as np
import torch


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Raw BF16 bits -> exact float64 values."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, dtype=np.float64))
    out = np.full(a.shape, 2.0 ** -133)
    normal = a >= 2.0 ** -126
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(normal, a, 1.0)))
    out[normal] = np.exp2(e[normal] - 7)
    return out


def gamma(n: int) -> float:
    u = 2.0 ** -24
    return n * u / (1.0 - n * u)


def abs_dot(x_bits: np.ndarray, W_bits: np.ndarray) -> np.ndarray:
    """sum_k |x[m,k]| |W[n,k]| in float64, shape [M, N]."""
    xa = torch.from_numpy(np.abs(bits_to_f64(x_bits)))
    wa = torch.from_numpy(np.abs(bits_to_f64(W_bits)))
    xa = torch.nan_to_num(xa, nan=0.0, posinf=0.0)
    wa = torch.nan_to_num(wa, nan=0.0, posinf=0.0)
    return (xa @ wa.T).numpy()


def compare(y_gpu_bits, y_ref_bits, x_bits, W_bits, *, tight: bool = True,
            cosine: bool = True) -> dict:
    """Check one GEMM result; returns a report dict with ``ok`` and the worst cases.

    ``cosine=False`` drops the per-row cosine from ``ok``; only hand-made cases
    whose exact sum is lost to any FP32 accumulation (catastrophic
    cancellation of terms 2^100 apart) use it."""
    y_gpu_bits = np.asarray(y_gpu_bits, dtype=np.uint16)
    y_ref_bits = np.asarray(y_ref_bits, dtype=np.uint16)
    g = bits_to_f64(y_gpu_bits)
    r = bits_to_f64(y_ref_bits)
    xv = bits_to_f64(x_bits)
    wv = bits_to_f64(W_bits)
    K = xv.shape[1]
    fin_x = np.isfinite(xv)
    fin_w = np.isfinite(wv)
    max_x = float(np.max(np.abs(xv[fin_x]), initial=0.0))
    max_w = float(np.max(np.abs(wv[fin_w]), initial=0.0))

    rep = {"ok": True, "n": int(r.size), "K": int(K)}
    ref_fin = np.isfinite(r)
    # non-finite references: same kind
    bad_kind = (~ref_fin) & ~((np.isnan(r) & np.isnan(g)) | (r == g))
    # finite references must get finite results
    bad_kind |= ref_fin & ~np.isfinite(g)
    rep["bad_kind"] = int(bad_kind.sum())

    with np.errstate(invalid="ignore"):
        diff = np.where(ref_fin & np.isfinite(g), np.abs(g - r), 0.0)
    ns_tol = 2.0 * ulp_bf16(r) + 1e-3 * np.sqrt(K) * max_x * max_w
    ns_bad = ref_fin & (diff > ns_tol)
    rep["ns_violations"] = int(ns_bad.sum())
    rep["max_err_over_ns_tol"] = float(np.max(np.where(ref_fin, diff / ns_tol, 0.0), initial=0.0))

    if tight:
        e = gamma(max(K - 1, 0)) * abs_dot(x_bits, W_bits) + K * 2.0 ** -150
        t_tol = 2.0 * ulp_bf16(np.abs(r) + e) + e
        t_bad = ref_fin & (diff > t_tol)
        rep["tight_violations"] = int(t_bad.sum())
        rep["max_err_over_tight_tol"] = float(
            np.max(np.where(ref_fin, diff / t_tol, 0.0), initial=0.0))
    else:
        t_bad = np.zeros_like(ns_bad)

    # the pages' SM90 bound, informational
    p_tol = 7.5e-5 + 2.0 ** -8 * np.abs(r)
    rep["pages_sm90_bound_violations"] = int((ref_fin & (diff > p_tol)).sum())
    rep["bitwise_equal_frac"] = float(np.mean(y_gpu_bits == y_ref_bits)) if r.size else 1.0

    # cosine per output row, finite entries only
    cos_min = 1.0
    for m in range(r.shape[0]):
        sel = ref_fin[m] & np.isfinite(g[m])
        a, b = g[m][sel], r[m][sel]
        na, nb = np.linalg.norm(a), np.linalg.norm(b)
        if na == 0.0 and nb == 0.0:
            c = 1.0
        elif na == 0.0 or nb == 0.0:
            c = 0.0
        else:
            c = float(np.dot(a, b) / (na * nb))
        cos_min = min(cos_min, c)
    rep["cosine_min"] = cos_min

    rep["ok"] = bool(rep["bad_kind"] == 0 and not ns_bad.any() and not t_bad.any()
                     and (cos_min >= 0.99999 or not cosine))
    return rep


def f32_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Raw FP32 bits (uint32) -> exact float64 values."""
    return np.asarray(b, dtype=np.uint32).view(np.float32).astype(np.float64)


def ulp_f32(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, dtype=np.float64))
    out = np.full(a.shape, 2.0 ** -149)
    normal = a >= 2.0 ** -126
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(normal, a, 1.0)))
    out[normal] = np.exp2(e[normal] - 23)
    return out


def compare_f32(y_gpu_bits, y_ref_bits, x_bits, W_bits) -> dict:
    """Check an FP32-output GEMM against the oracle's FP32 reference (bits as uint32)."""
    g = f32_bits_to_f64(y_gpu_bits)
    r = f32_bits_to_f64(y_ref_bits)
    K = np.asarray(x_bits).shape[1]
    rep = {"ok": True, "n": int(r.size), "K": int(K)}
    ref_fin = np.isfinite(r)
    bad_kind = (~ref_fin) & ~((np.isnan(r) & np.isnan(g)) | (r == g))
    bad_kind |= ref_fin & ~np.isfinite(g)
    rep["bad_kind"] = int(bad_kind.sum())
    with np.errstate(invalid="ignore"):
        diff = np.where(ref_fin & np.isfinite(g), np.abs(g - r), 0.0)
    e = gamma(max(K - 1, 0)) * abs_dot(x_bits, W_bits) + K * 2.0 ** -150
    tol = e + 0.5 * ulp_f32(r)
    bad = ref_fin & (diff > tol)
    rep["violations"] = int(bad.sum())
    rep["max_err_over_tol"] = float(np.max(np.where(ref_fin, diff / tol, 0.0), initial=0.0))
    rep["bitwise_equal_frac"] = float(np.mean(np.asarray(y_gpu_bits) == np.asarray(y_ref_bits))) \
        if r.size else 1.0
    cos_min = 1.0
    for m in range(r.shape[0]):
        sel = ref_fin[m] & np.isfinite(g[m])
        a, b = g[m][sel], r[m][sel]
        na, nb = np.linalg.norm(a), np.linalg.norm(b)
        c = 1.0 if (na == 0.0 and nb == 0.0) else (0.0 if na == 0.0 or nb == 0.0
                                                    else float(np.dot(a, b) / (na * nb)))
        cos_min = min(cos_min, c)
    rep["cosine_min"] = cos_min
    rep["ok"] = bool(rep["bad_kind"] == 0 and not bad.any() and cos_min >= 0.99999)
    return rep
