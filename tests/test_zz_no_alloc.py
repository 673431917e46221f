"""The split-K entry point that allocates nothing (collected last on purpose).

Some callers cannot allocate device memory when they run a GEMM: code under a
memory manager that owns all of the GPU's memory, plugins or embedded runtimes
that may not grow their footprint after start-up, or loops where a possibly
synchronizing cudaMalloc is not allowed.  sgemm_bf16_skinny_splitk_noalloc
serves them: its split-K partial sums live in a fixed 4 MiB device array inside
the library instead of allocated scratch.

Each case calls it through the C ABI twice in a row, with different inputs, and
checks each output against the CPU oracle (within the tolerance every parity
test here uses) and bitwise against sgemm_bf16_skinny_ex run with the plan the
call documents (sgemm_splitk_noalloc_plan).  A stale partial sum left by the
first call would break the second comparison.  The shapes reach every kind of
selected plan the call substitutes.  It also checks that a problem too large
for the fixed array is refused, and, in a fresh process, that a first call made
while the stream is capturing is refused without enqueuing anything.  It must
pass alone in a fresh process and after the rest of the suite.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
import oracle
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(M, N, K, seed):
    x = synth.normal_bf16((M, K), synth.X_STD, seed=seed).to("cuda")
    W = synth.normal_bf16((N, K), synth.W_STD, seed=seed + 1).to("cuda")
    return x, W


# (M, N, K, split): the first four as before; (4096, 4096) at M = 3 and 4 and
# (12576, 4096) at M = 4 select tensor-core plans that the call replaces
@pytest.mark.parametrize("M,N,K,split", [(1, 4096, 8192, 4), (4, 1000, 4096, 3),
                                         (2, 2048, 4096, 2), (3, 517, 1536, 5),
                                         (3, 4096, 4096, 2), (4, 4096, 4096, 4),
                                         (4, 12576, 4096, 2), (8, 4096, 1024, 3)])
def test_no_alloc_matches_oracle_and_regular_call_on_two_calls(M, N, K, split):
    assert torch.cuda.is_available()
    sk.load()
    st, plan = sk.sgemm_splitk_noalloc_plan(N, K, M, split)
    assert st == sk.SGEMM_OK, (st, plan)
    (xa, Wa), (xb, Wb) = _inputs(M, N, K, 900 + M), _inputs(M, N, K, 950 + M)
    ya = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    yb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    # two calls in a row on the no-allocation entry point
    sk.sgemm_bf16_skinny_splitk_noalloc(xa, Wa, ya, split_k=split)
    sk.sgemm_bf16_skinny_splitk_noalloc(xb, Wb, yb, split_k=split)
    torch.cuda.synchronize()
    rows = torch.arange(0, N, max(1, N // 600))  # the oracle on a row sample for large N
    for x, W, y in ((xa, Wa, ya), (xb, Wb, yb)):
        reg = sk.sgemm_bf16_skinny_ex(x, W, plan=plan)  # the regular call, same plan
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), reg.view(torch.int16)), plan
        xs, Ws = synth.bits(x.cpu()), synth.bits(W[rows.cuda()].cpu())
        rep = compare(synth.bits(y.cpu())[:, rows.numpy()], oracle.skinny_gemm(xs, Ws), xs, Ws)
        assert rep["ok"], rep


def test_no_alloc_refuses_problems_larger_than_its_scratch():
    lib = sk.load()
    M, N, K, split = 4, 77440, 4096, 4  # 4*4*77440*4 bytes > 4 MiB
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.sgemm_bf16_skinny_splitk_noalloc(x.data_ptr(), K, W.data_ptr(), y.data_ptr(), N,
                                              M, N, K, split, None)
    assert st == sk.SGEMM_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(sk.SgemmError):
        sk.sgemm_bf16_skinny_splitk_noalloc(x, W, y, split_k=split)


FIRST_CALL_IN_CAPTURE = r"""
import sys, torch
sys.path.insert(0, {root!r})
import bf16_skinny_gemm_gb300 as sk
lib = sk.load()
x = torch.ones((1, 1024), dtype=torch.bfloat16, device="cuda")
W = torch.ones((512, 1024), dtype=torch.bfloat16, device="cuda")
y = torch.zeros((1, 512), dtype=torch.bfloat16, device="cuda")
torch.cuda.synchronize()
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.stream(s):
    with torch.cuda.graph(g, stream=s):
        st = lib.sgemm_bf16_skinny_splitk_noalloc(x.data_ptr(), 1024, W.data_ptr(), y.data_ptr(),
                                                  512, 1, 512, 1024, 2, s.cuda_stream)
assert st == sk.SGEMM_ERR_INVALID_ARG, st
# outside capture the set-up happens and the call works; then it may be captured
sk.sgemm_bf16_skinny_splitk_noalloc(x, W, y, split_k=2)
torch.cuda.synchronize()
assert torch.all(y == 1024.0), y
y.zero_()
g2 = torch.cuda.CUDAGraph()
with torch.cuda.stream(s):
    with torch.cuda.graph(g2, stream=s):
        sk.sgemm_bf16_skinny_splitk_noalloc(x, W, y, split_k=2, stream=s)
g2.replay()
torch.cuda.synchronize()
assert torch.all(y == 1024.0), y
print("ok")
"""


def test_first_call_during_capture_is_refused_in_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", FIRST_CALL_IN_CAPTURE.format(root=ROOT)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
