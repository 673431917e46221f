"""GB300 (sm_103a) BF16 skinny GEMM: ``y[M,N] = x[M,K] @ W[N,K]^T`` for M = 1..8.

A thin ctypes binding over the C ABI of ``libsgemm_skinny.so`` (declared in
``include/sgemm_skinny.h``).  The functions keep the C names and only marshal
arguments: torch tensors become device pointers, row strides and the current
CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and a missing library raises.

PyTorch is used here only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

__all__ = [
    "SgemmError", "Plan", "Pair", "load", "library_path",
    "sgemm_bf16_skinny", "sgemm_bf16_skinny_ex", "sgemm_bf16_skinny_batched",
    "sgemm_bf16_skinny_batched_ex", "sgemm_plan_select", "sgemm_plan_count", "sgemm_plan_get",
    "sgemm_plan_check", "sgemm_init", "sgemm_status_string", "sgemm_version",
    "sgemm_bf16_skinny_splitk_noalloc", "sgemm_splitk_noalloc_plan", "NOALLOC_SCRATCH_BYTES",
    "sgemm_bf16_rescale",
    "sgemm_bf16_skinny_rescale_ex", "sgemm_bf16_skinny_f32out_ex",
    "SGEMM_OK", "SGEMM_ERR_INVALID_ARG", "SGEMM_ERR_UNSUPPORTED_SHAPE", "SGEMM_ERR_MISALIGNED",
    "SGEMM_ERR_UNSUPPORTED_DEVICE", "SGEMM_ERR_NO_WORKSPACE", "SGEMM_ERR_CUDA", "MAX_BATCH",
    "SGEMM_VARIANT_LDG", "SGEMM_VARIANT_LDG_MIXFMA", "SGEMM_VARIANT_MMA", "SGEMM_VARIANT_LDG_FFMA2",
    "SGEMM_VARIANT_LDGX_MIXFMA", "SGEMM_VARIANT_LDGX_FFMA2", "SGEMM_VARIANT_LDG_MMA",
    "SGEMM_VARIANT_LDG_CLUSTER",
    "SGEMM_VARIANT_TC05", "SGEMM_FLAG_PDL",
    "SGEMM_FLAG_TEST_STALL", "sgemm_device_errors",
    "SGEMM_FLAG_WEIGHTS_READONLY",
]

SGEMM_OK = 0
SGEMM_ERR_INVALID_ARG = 1
SGEMM_ERR_UNSUPPORTED_SHAPE = 2
SGEMM_ERR_MISALIGNED = 3
SGEMM_ERR_UNSUPPORTED_DEVICE = 4
SGEMM_ERR_NO_WORKSPACE = 5
SGEMM_ERR_CUDA = 6
MAX_BATCH = 8
SGEMM_VARIANT_LDG = 0
SGEMM_VARIANT_LDG_MIXFMA = 1
SGEMM_VARIANT_MMA = 2
SGEMM_VARIANT_LDG_FFMA2 = 5
SGEMM_VARIANT_LDGX_MIXFMA = 6
SGEMM_VARIANT_LDGX_FFMA2 = 7
SGEMM_VARIANT_LDG_MMA = 9
SGEMM_VARIANT_TC05 = 10
SGEMM_VARIANT_LDG_CLUSTER = 11
SGEMM_FLAG_TEST_STALL = 4
SGEMM_FLAG_PDL = 1
SGEMM_FLAG_WEIGHTS_READONLY = 2


class Plan(ctypes.Structure):
    """Mirror of ``sgemm_plan_t``."""
    _fields_ = [(name, ctypes.c_int) for name in (
        "variant", "threads", "rows_per_warp", "lanes_per_row", "k_unroll", "vec_bytes",
        "split_k", "stages", "ctas_per_sm", "id")]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}

    def copy(self, **changes) -> "Plan":
        p = Plan(**self.as_dict())
        for k, v in changes.items():
            setattr(p, k, v)
        return p

    def __repr__(self) -> str:
        return "Plan(" + ", ".join(f"{k}={v}" for k, v in self.as_dict().items()) + ")"


class Pair(ctypes.Structure):
    """Mirror of ``sgemm_pair_t``."""
    _fields_ = [("x", ctypes.c_void_p), ("W", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("ldx", ctypes.c_longlong), ("ldy", ctypes.c_longlong)]


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        msg = sgemm_status_string(status) if _lib is not None else f"status {status}"
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return os.environ.get("SGEMM_SKINNY_LIB", LIB_PATH)


def load() -> ctypes.CDLL:
    """Load ``libsgemm_skinny.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, ll, ci = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int
        lib.sgemm_bf16_skinny.argtypes = [vp, vp, vp, ci, ci, ci, vp]
        lib.sgemm_bf16_skinny.restype = ci
        cu = ctypes.c_uint
        lib.sgemm_bf16_skinny_ex.argtypes = [vp, ll, vp, vp, ll, ci, ci, ci,
                                             ctypes.POINTER(Plan), cu, vp]
        lib.sgemm_bf16_skinny_ex.restype = ci
        lib.sgemm_bf16_skinny_rescale_ex.argtypes = [vp, ll, vp, vp, ll, ci, ci, ci, vp, ll, ll,
                                                     ctypes.c_float, ctypes.POINTER(Plan), cu, vp]
        lib.sgemm_bf16_skinny_rescale_ex.restype = ci
        lib.sgemm_bf16_skinny_f32out_ex.argtypes = [vp, ll, vp, vp, ll, ci, ci, ci,
                                                    ctypes.POINTER(Plan), cu, vp]
        lib.sgemm_bf16_skinny_f32out_ex.restype = ci
        lib.sgemm_bf16_skinny_batched.argtypes = [ctypes.POINTER(Pair), ci, ci, ci, ci, vp]
        lib.sgemm_bf16_skinny_batched.restype = ci
        lib.sgemm_bf16_skinny_batched_ex.argtypes = [ctypes.POINTER(Pair), ci, ci, ci, ci,
                                                     ctypes.POINTER(Plan), cu, vp]
        lib.sgemm_bf16_skinny_batched_ex.restype = ci
        lib.sgemm_plan_select.argtypes = [ci, ci, ci]
        lib.sgemm_plan_select.restype = Plan
        lib.sgemm_plan_count.argtypes = []
        lib.sgemm_plan_count.restype = ci
        lib.sgemm_plan_get.argtypes = [ci, ctypes.POINTER(Plan)]
        lib.sgemm_plan_get.restype = ci
        lib.sgemm_plan_check.argtypes = [ctypes.POINTER(Plan), ci, ci, ci]
        lib.sgemm_plan_check.restype = ci
        lib.sgemm_init.argtypes = []
        lib.sgemm_init.restype = ci
        lib.sgemm_status_string.argtypes = [ci]
        lib.sgemm_status_string.restype = ctypes.c_char_p
        lib.sgemm_bf16_skinny_splitk_noalloc.argtypes = [vp, ll, vp, vp, ll, ci, ci, ci, ci, vp]
        lib.sgemm_bf16_skinny_splitk_noalloc.restype = ci
        lib.sgemm_splitk_noalloc_plan.argtypes = [ci, ci, ci, ci, ctypes.POINTER(Plan),
                                                  ctypes.POINTER(Plan)]
        lib.sgemm_splitk_noalloc_plan.restype = ci
        lib.sgemm_bf16_rescale.argtypes = [vp, ll, vp, ll, ctypes.c_float, cu, vp]
        lib.sgemm_bf16_rescale.restype = ci
        lib.sgemm_device_errors.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.sgemm_device_errors.restype = ci
        lib.sgemm_version.argtypes = []
        lib.sgemm_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, what: str):
    if status != SGEMM_OK:
        raise SgemmError(status, what)


def _bf16_2d(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D torch.bfloat16 tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be on a CUDA device")
    if t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")


def _problem(x, W, y):
    _bf16_2d(x, "x")
    _bf16_2d(W, "W")
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K or (W.stride(0) != K and N > 1):
        raise ValueError(f"W must be a contiguous [N, {K}] tensor, got {tuple(W.shape)}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _bf16_2d(y, "y")
    if tuple(y.shape) != (M, N):
        raise ValueError(f"y must be [{M}, {N}], got {tuple(y.shape)}")
    return M, N, K, y


def sgemm_bf16_skinny(x: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """``y = x @ W.T`` for contiguous x [M,K], W [N,K]; returns y [M,N]."""
    M, N, K, y = _problem(x, W, y)
    if x.stride(0) != K and M > 1 or y.stride(0) != N and M > 1:
        raise ValueError("sgemm_bf16_skinny wants contiguous x and y; use sgemm_bf16_skinny_ex")
    _check(load().sgemm_bf16_skinny(x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K,
                                    _stream(stream)), "sgemm_bf16_skinny")
    return y


def sgemm_bf16_skinny_ex(x: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None,
                         plan: Plan | None = None, flags: int = 0, stream=None) -> torch.Tensor:
    """Like :func:`sgemm_bf16_skinny` with strided x / y rows, an optional plan
    and launch flags (``SGEMM_FLAG_*``)."""
    M, N, K, y = _problem(x, W, y)
    ldx = x.stride(0) if M > 1 else K
    ldy = y.stride(0) if M > 1 else N
    _check(load().sgemm_bf16_skinny_ex(x.data_ptr(), ldx, W.data_ptr(), y.data_ptr(), ldy,
                                       M, N, K, ctypes.byref(plan) if plan is not None else None,
                                       int(flags), _stream(stream)), "sgemm_bf16_skinny_ex")
    return y


def sgemm_bf16_skinny_rescale_ex(x: torch.Tensor, W: torch.Tensor, y: torch.Tensor,
                                 x_next: torch.Tensor, scale: float, plan: Plan | None = None,
                                 flags: int = 0, stream=None) -> torch.Tensor:
    """One decode-chain GEMM with the elementwise step fused into its epilogue:
    ``y = x @ W.T`` and ``x_next[m, k] = bf16(float(y[m, k % N]) * scale)`` for every
    column k of x_next ([M, n_next] BF16, its own buffer).  Returns y."""
    M, N, K, y = _problem(x, W, y)
    _bf16_2d(x_next, "x_next")
    if x_next.shape[0] != M:
        raise ValueError(f"x_next must have {M} rows, got {x_next.shape[0]}")
    n_next = x_next.shape[1]
    ldx = x.stride(0) if M > 1 else K
    ldy = y.stride(0) if M > 1 else N
    ldn = x_next.stride(0) if M > 1 else n_next
    _check(load().sgemm_bf16_skinny_rescale_ex(
        x.data_ptr(), ldx, W.data_ptr(), y.data_ptr(), ldy, M, N, K, x_next.data_ptr(), ldn,
        n_next, float(scale), ctypes.byref(plan) if plan is not None else None, int(flags),
        _stream(stream)), "sgemm_bf16_skinny_rescale_ex")
    return y


def sgemm_bf16_skinny_f32out_ex(x: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None,
                                plan: Plan | None = None, flags: int = 0,
                                stream=None) -> torch.Tensor:
    """``y = x @ W.T`` with FP32 outputs (y: float32 [M, N], row-strided allowed)."""
    _bf16_2d(x, "x")
    _bf16_2d(W, "W")
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K or (W.stride(0) != K and N > 1):
        raise ValueError(f"W must be a contiguous [N, {K}] tensor, got {tuple(W.shape)}")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if y.dtype != torch.float32 or y.dim() != 2 or tuple(y.shape) != (M, N) or y.stride(1) != 1:
        raise ValueError(f"y must be a float32 [{M}, {N}] tensor with unit column stride")
    ldx = x.stride(0) if M > 1 else K
    ldy = y.stride(0) if M > 1 else N
    _check(load().sgemm_bf16_skinny_f32out_ex(
        x.data_ptr(), ldx, W.data_ptr(), y.data_ptr(), ldy, M, N, K,
        ctypes.byref(plan) if plan is not None else None, int(flags), _stream(stream)),
        "sgemm_bf16_skinny_f32out_ex")
    return y


def _pairs(items):
    if not 1 <= len(items) <= MAX_BATCH:
        raise ValueError(f"batch must be 1..{MAX_BATCH}")
    arr = (Pair * len(items))()
    shape = None
    outs = []
    for i, it in enumerate(items):
        x, W = it[0], it[1]
        y = it[2] if len(it) > 2 else None
        M, N, K, y = _problem(x, W, y)
        if shape is None:
            shape = (M, N, K)
        elif shape != (M, N, K):
            raise ValueError("every item of a batched call must have the same (M, N, K)")
        arr[i].x = x.data_ptr()
        arr[i].W = W.data_ptr()
        arr[i].y = y.data_ptr()
        arr[i].ldx = x.stride(0) if M > 1 else K
        arr[i].ldy = y.stride(0) if M > 1 else N
        outs.append(y)
    return arr, shape, outs


def sgemm_bf16_skinny_batched(items, stream=None) -> list:
    """One launch for ``[(x_i, W_i[, y_i]), ...]`` of one shape; returns the y_i."""
    arr, (M, N, K), outs = _pairs(items)
    _check(load().sgemm_bf16_skinny_batched(arr, len(items), M, N, K, _stream(stream)),
           "sgemm_bf16_skinny_batched")
    return outs


def sgemm_bf16_skinny_batched_ex(items, plan: Plan | None = None, flags: int = 0,
                                 stream=None) -> list:
    """:func:`sgemm_bf16_skinny_batched` with an explicit plan and launch flags."""
    arr, (M, N, K), outs = _pairs(items)
    _check(load().sgemm_bf16_skinny_batched_ex(arr, len(items), M, N, K,
                                               ctypes.byref(plan) if plan is not None else None,
                                               int(flags), _stream(stream)),
           "sgemm_bf16_skinny_batched_ex")
    return outs


def sgemm_bf16_rescale(y: torch.Tensor, x: torch.Tensor, scale: float, flags: int = 0,
                       stream=None) -> torch.Tensor:
    """``x.view(-1)[k] = bf16(float(y.view(-1)[k % y.numel()]) * scale)`` on the GPU: the
    elementwise step between two GEMMs of a decode chain.  Returns x."""
    for t, name in ((y, "y"), (x, "x")):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    _check(load().sgemm_bf16_rescale(y.data_ptr(), y.numel(), x.data_ptr(), x.numel(),
                                     float(scale), int(flags), _stream(stream)),
           "sgemm_bf16_rescale")
    return x


NOALLOC_SCRATCH_BYTES = 4 << 20


def sgemm_bf16_skinny_splitk_noalloc(x: torch.Tensor, W: torch.Tensor,
                                     y: torch.Tensor | None = None, split_k: int = 2,
                                     stream=None) -> torch.Tensor:
    """Split-K ``y = x @ W.T`` that allocates nothing on the device.

    For callers that may not allocate device memory when they run the GEMM
    (a memory manager that owns the GPU's memory, a plugin with a fixed
    footprint, a loop where a synchronizing allocation is not allowed).  The
    partial sums live in a fixed 4 MiB array inside the library, shared by all
    calls on a device: calls that overlap on the GPU race, and the first call
    on a device (which looks the array up) should come before stream capture.
    ``y`` must be given for the call itself to allocate nothing (otherwise this
    wrapper creates it with torch).  Results equal ``sgemm_bf16_skinny_ex`` with
    the plan :func:`sgemm_splitk_noalloc_plan` returns.
    """
    M, N, K, y = _problem(x, W, y)
    need = int(split_k) * M * N * 4
    if need > NOALLOC_SCRATCH_BYTES:
        raise SgemmError(SGEMM_ERR_UNSUPPORTED_SHAPE,
                         f"sgemm_bf16_skinny_splitk_noalloc: split_k*M*N*4 = {need} bytes of "
                         f"partial sums exceed the fixed {NOALLOC_SCRATCH_BYTES}-byte scratch")
    ldx = x.stride(0) if M > 1 else K
    ldy = y.stride(0) if M > 1 else N
    _check(load().sgemm_bf16_skinny_splitk_noalloc(x.data_ptr(), ldx, W.data_ptr(), y.data_ptr(),
                                                   ldy, M, N, K, int(split_k), _stream(stream)),
           "sgemm_bf16_skinny_splitk_noalloc")
    return y


def sgemm_splitk_noalloc_plan(N: int, K: int, M: int, split_k: int,
                              selected: Plan | None = None) -> tuple[int, Plan]:
    """(status, plan): the plan :func:`sgemm_bf16_skinny_splitk_noalloc` runs for
    this problem, from ``selected`` (default: the selected plan) with split_k
    splits through scratch memory (host-only)."""
    out = Plan()
    st = load().sgemm_splitk_noalloc_plan(int(N), int(K), int(M), int(split_k),
                                          ctypes.byref(selected) if selected is not None else None,
                                          ctypes.byref(out))
    return st, out


def sgemm_plan_select(N: int, K: int, M: int) -> Plan:
    """The plan the library uses for (N, K, M) (host-only)."""
    return load().sgemm_plan_select(int(N), int(K), int(M))


def sgemm_plan_count() -> int:
    return load().sgemm_plan_count()


def sgemm_plan_get(index: int) -> Plan:
    p = Plan()
    _check(load().sgemm_plan_get(int(index), ctypes.byref(p)), "sgemm_plan_get")
    return p


def sgemm_plan_check(plan: Plan, M: int, N: int, K: int) -> int:
    """Status a call with this plan and shape would get from its plan check."""
    return load().sgemm_plan_check(ctypes.byref(plan), int(M), int(N), int(K))


def sgemm_init() -> None:
    """Allocate the split-K scratch of the current device (before graph capture)."""
    _check(load().sgemm_init(), "sgemm_init")


def sgemm_device_errors() -> int:
    """Read and clear the device error word of the current device (synchronous).
    Bit 0: a kernel gave up a bounded wait for its data and wrote NaN outputs."""
    v = ctypes.c_int(0)
    _check(load().sgemm_device_errors(ctypes.byref(v)), "sgemm_device_errors")
    return v.value


def sgemm_status_string(status: int) -> str:
    return load().sgemm_status_string(int(status)).decode()


def sgemm_version() -> str:
    return load().sgemm_version().decode()
