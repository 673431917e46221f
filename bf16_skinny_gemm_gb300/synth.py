"""Seeded synthetic BF16 inputs for the skinny GEMM.

This module only draws numbers: it holds none of the GEMM's arithmetic and is
the one piece of code that both the GPU path's tests/benchmark and the CPU
oracle's tests use.  Values are drawn in float32 with a seeded torch generator
and converted to BF16 by PyTorch (round-to-nearest-even).

Input families follow vLLM PR #65306 ("Add SM90 skinny GEMM plans for the BF16
decode projections", Validation), which checks the kernel on "normal, outlier
and scaled/sparse inputs":

- ``normal``       N(0, std^2)
- ``outlier``      normal, with 1 in 256 entries replaced by +-2^10 * |N(0,1)| * std
- ``scaled_up``    normal * 2^20
- ``scaled_down``  normal * 2^-20
- ``sparse``       normal with 90 % of the entries set to zero

The workload scales (x ~ N(0,1), W ~ N(0, 0.02^2), pair weights ~ N(0, 0.05^2))
are the decode-projection workloads the pages measure on; the pages publish no
value distribution, so these are synthetic stand-ins for real activations and
checkpoint weights.
"""
from __future__ import annotations

import numpy as np
import torch

FAMILIES = ("normal", "outlier", "scaled_up", "scaled_down", "sparse")

# scale of the decode workloads (x ~ N(0,1), W ~ N(0, 0.02^2)); pairs use 0.05
X_STD = 1.0
W_STD = 0.02
PAIR_W_STD = 0.05


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float = 1.0, seed: int = 0, device="cpu") -> torch.Tensor:
    """BF16 tensor of N(0, std^2) draws; same seed and device give the same bits."""
    g = _gen(seed, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def family_bf16(shape, kind: str, std: float = 1.0, seed: int = 0, device="cpu") -> torch.Tensor:
    """BF16 tensor from one of :data:`FAMILIES`."""
    if kind not in FAMILIES:
        raise ValueError(f"unknown input family {kind!r}")
    g = _gen(seed, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32) * std
    if kind == "outlier":
        pick = torch.rand(tuple(shape), generator=g, device=device) < (1.0 / 256.0)
        sign = torch.where(torch.rand(tuple(shape), generator=g, device=device) < 0.5, -1.0, 1.0)
        t = torch.where(pick, sign * 1024.0 * std * t.abs().clamp_min(0.25), t)
    elif kind == "scaled_up":
        t = t * (2.0 ** 20)
    elif kind == "scaled_down":
        t = t * (2.0 ** -20)
    elif kind == "sparse":
        keep = torch.rand(tuple(shape), generator=g, device=device) < 0.1
        t = t * keep
    return t.to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw BF16 bit patterns (uint16 numpy array, on the host) of a BF16 tensor."""
    if t.dtype != torch.bfloat16:
        raise TypeError(f"expected a bfloat16 tensor, got {t.dtype}")
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, device="cpu") -> torch.Tensor:
    """BF16 tensor holding the given raw bit patterns."""
    a = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
