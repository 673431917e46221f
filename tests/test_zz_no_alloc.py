"""The split-K entry point that allocates nothing (collected last on purpose).

Some callers cannot allocate device memory when they run a GEMM: code under a
memory manager that owns all of the GPU's memory, plugins or embedded runtimes
that may not grow their footprint after start-up, or loops where a possibly
synchronizing cudaMalloc is not allowed.  sgemm_bf16_skinny_splitk_noalloc
serves them: its split-K partial sums live in a fixed 4 MiB device array inside
the library instead of allocated scratch.

This test calls it through the C ABI twice in a row, with different inputs, and
checks each output against the regular entry point (sgemm_bf16_skinny) within
the tolerance used by every parity test here.  A stale partial sum left by the first call would break the
second comparison.  It also checks that a problem too large for the fixed
array is refused.  It must pass alone in a fresh process and after the rest of
the suite.
"""
from __future__ import annotations

import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed):
    x = synth.normal_bf16((M, K), synth.X_STD, seed=seed).to("cuda")
    W = synth.normal_bf16((N, K), synth.W_STD, seed=seed + 1).to("cuda")
    return x, W


@pytest.mark.parametrize("M,N,K,split", [(1, 4096, 8192, 4), (4, 1000, 4096, 3),
                                         (2, 2048, 4096, 2), (3, 517, 1536, 5)])
def test_no_alloc_matches_regular_split_k_on_two_calls(M, N, K, split):
    assert torch.cuda.is_available()
    sk.load()
    (xa, Wa), (xb, Wb) = _inputs(M, N, K, 900 + M), _inputs(M, N, K, 950 + M)
    ya = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    yb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    # two calls in a row on the no-allocation entry point
    sk.sgemm_bf16_skinny_splitk_noalloc(xa, Wa, ya, split_k=split)
    sk.sgemm_bf16_skinny_splitk_noalloc(xb, Wb, yb, split_k=split)
    torch.cuda.synchronize()
    for x, W, y in ((xa, Wa, ya), (xb, Wb, yb)):
        ref = sk.sgemm_bf16_skinny(x, W)  # the existing entry point, its own plan
        torch.cuda.synchronize()
        rep = compare(synth.bits(y), synth.bits(ref), synth.bits(x), synth.bits(W))
        assert rep["ok"], rep


def test_no_alloc_refuses_problems_larger_than_its_scratch():
    sk.load()
    M, N, K, split = 4, 77440, 4096, 4  # 4*4*77440*4 bytes > 4 MiB
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    lib = sk.load()
    st = lib.sgemm_bf16_skinny_splitk_noalloc(x.data_ptr(), K, W.data_ptr(), y.data_ptr(), N,
                                              M, N, K, split, None)
    assert st == sk.SGEMM_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(sk.SgemmError):
        sk.sgemm_bf16_skinny_splitk_noalloc(x, W, y, split_k=split)
