"""CPU oracle for the BF16 skinny GEMM ``y[M,N] = x[M,K] @ W[N,K]^T``.

TEST INFRASTRUCTURE ONLY.  The test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are its only users; the GPU library never
imports, calls or links anything here, and nothing here imports the GPU
library.

The arithmetic lives in ``skinny_oracle.c`` (plain C, exact fixed-point
accumulation, one round-to-nearest-even to BF16 at the end; the header of that
file states the definition and cites the pages it follows).  This module only
builds it with gcc, loads it with ctypes and marshals numpy arrays of raw BF16
bits (``uint16``); the FP32-output form returns FP32 bit patterns (``uint32``).

Parity status: pinned.  ``tests/test_oracle_pins.py`` checks it against an
independent brute-force rounding of exact rational sums, hand-derived closed
forms (``tests/golden/closed_forms.txt``) and exact invariants, and shows that
deliberately planted mistakes in a copy of the C source fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "skinny_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_skinny.so")


def compile_library(src: str, out: str) -> str:
    """gcc -O2 a C source file into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-fPIC", "-shared", "-pthread", "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle_skinny.so`` if stale."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE))
    if force or stale:
        compile_library(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"oracle wants raw BF16 bits as uint16, got {a.dtype}")
    return a


class Oracle:
    """One loaded build of the oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64p = ctypes.POINTER(ctypes.c_int64)
        ip = ctypes.POINTER(ctypes.c_int)
        ll = ctypes.c_longlong
        ci = ctypes.c_int
        lib.oracle_bf16_skinny_gemm.argtypes = [u16p, ll, u16p, ll, u16p, ll, ci, ci, ci, ci]
        lib.oracle_bf16_skinny_gemm.restype = ci
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.oracle_bf16_skinny_gemm_f32.argtypes = [u16p, ll, u16p, ll, u32p, ll, ci, ci, ci, ci]
        lib.oracle_bf16_skinny_gemm_f32.restype = ci
        lib.oracle_exact_dot.argtypes = [u16p, u16p, ci, i64p, ip, ip]
        lib.oracle_exact_dot.restype = ctypes.c_uint16
        lib.oracle_cores.restype = ci
        lib.oracle_acc_digits.restype = ci
        lib.oracle_acc_bias.restype = ci
        self._lib = lib
        self.path = lib_path

    def cores(self) -> int:
        """CPUs in this process's affinity mask (the default thread count)."""
        return self._lib.oracle_cores()

    def skinny_gemm(self, x_bits, W_bits, threads: int = 0, return_threads: bool = False):
        """``y_ref`` bits [M,N] for x bits [M,K] and W bits [N,K].

        Every element is RNE_bf16 of the exact dot product of a row of x and a
        row of W.  ``threads <= 0`` uses every CPU of the affinity mask; the
        result does not depend on the thread count.
        """
        x = _u16(x_bits)
        W = _u16(W_bits)
        if x.ndim != 2 or W.ndim != 2 or x.shape[1] != W.shape[1]:
            raise ValueError(f"shapes x{x.shape} W{W.shape} do not form x @ W^T")
        if x.strides[1] != 2 or x.strides[0] % 2:
            x = np.ascontiguousarray(x)
        if W.strides[1] != 2 or W.strides[0] % 2:
            W = np.ascontiguousarray(W)
        M, K = x.shape
        N = W.shape[0]
        y = np.zeros((M, N), dtype=np.uint16)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        used = self._lib.oracle_bf16_skinny_gemm(
            x.ctypes.data_as(u16p), max(x.strides[0] // 2, K),
            W.ctypes.data_as(u16p), max(W.strides[0] // 2, K),
            y.ctypes.data_as(u16p), N, M, N, K, int(threads))
        if used < 0:
            raise ValueError("oracle rejected its arguments")
        return (y, used) if return_threads else y

    def skinny_gemm_f32(self, x_bits, W_bits, threads: int = 0):
        """FP32 bit patterns (uint32) [M,N]: RNE_fp32 of each exact dot product."""
        x = np.ascontiguousarray(_u16(x_bits))
        W = np.ascontiguousarray(_u16(W_bits))
        if x.ndim != 2 or W.ndim != 2 or x.shape[1] != W.shape[1]:
            raise ValueError(f"shapes x{x.shape} W{W.shape} do not form x @ W^T")
        M, K = x.shape
        N = W.shape[0]
        y = np.zeros((M, N), dtype=np.uint32)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        used = self._lib.oracle_bf16_skinny_gemm_f32(
            x.ctypes.data_as(u16p), K, W.ctypes.data_as(u16p), K,
            y.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)), N, M, N, K, int(threads))
        if used < 0:
            raise ValueError("oracle rejected its arguments")
        return y

    def exact_dot(self, x_row, w_row):
        """Exact dot product of two BF16 rows.

        Returns ``(value, bf16_bits)``; ``value`` is a ``fractions.Fraction``
        for a finite sum, else one of ``"+inf"``, ``"-inf"``, ``"nan"``.
        """
        x = np.ascontiguousarray(_u16(x_row))
        w = np.ascontiguousarray(_u16(w_row))
        if x.shape != w.shape or x.ndim != 1:
            raise ValueError("exact_dot wants two equal-length 1-D rows")
        nd = self._lib.oracle_acc_digits()
        bias = self._lib.oracle_acc_bias()
        digits = (ctypes.c_int64 * nd)()
        sign = ctypes.c_int()
        special = ctypes.c_int()
        u16p = ctypes.POINTER(ctypes.c_uint16)
        bits = self._lib.oracle_exact_dot(x.ctypes.data_as(u16p), w.ctypes.data_as(u16p),
                                          x.shape[0], digits, ctypes.byref(sign),
                                          ctypes.byref(special))
        if special.value:
            return {1: "+inf", 2: "-inf", 3: "nan"}[special.value], int(bits)
        mag = 0
        for i in range(nd - 1, -1, -1):
            mag = (mag << 32) + int(digits[i])
        return Fraction(sign.value * mag, 1 << bias), int(bits)


_lock = threading.Lock()
_default = None


def default() -> Oracle:
    """The oracle built from ``skinny_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def skinny_gemm(x_bits, W_bits, threads: int = 0, return_threads: bool = False):
    """See :meth:`Oracle.skinny_gemm`."""
    return default().skinny_gemm(x_bits, W_bits, threads, return_threads)


def skinny_gemm_f32(x_bits, W_bits, threads: int = 0):
    """See :meth:`Oracle.skinny_gemm_f32`."""
    return default().skinny_gemm_f32(x_bits, W_bits, threads)


def exact_dot(x_row, w_row):
    """See :meth:`Oracle.exact_dot`."""
    return default().exact_dot(x_row, w_row)


def cores() -> int:
    """See :meth:`Oracle.cores`."""
    return default().cores()
