"""Failure detection on the GPU, without a GPU fault.

The TMA + tcgen05 kernel (SGEMM_VARIANT_TC05) waits on shared-memory mbarriers
for its copies and its tensor-core results.  Every wait is bounded (about
0.2 s); when one gives up, the kernel writes NaN to the outputs it owns, sets
bit 0 of the device error word, waits (bounded) for what it issued, frees its
tensor memory and returns, so the context stays usable.  The test-only launch
flag SGEMM_FLAG_TEST_STALL makes the kernel's producer issue no copies at all,
so the waits run out: nothing faults, traps or hangs.  The host reads the
status with sgemm_device_errors().  Both work splits are covered: the
persistent grid, and the cluster split, whose ranks push their partial tiles
to rank 0 (counted on an mbarrier that rank 0 waits on, bounded) and whose
CTAs that gave up take a second cluster barrier before they exit, so that no
partial tile lands in shared memory that has been released.
"""
from __future__ import annotations

import time

import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
import oracle
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare

pytestmark = pytest.mark.gpu


def _tc05(split):
    for i in range(sk.sgemm_plan_count()):
        p = sk.sgemm_plan_get(i)
        if p.variant == sk.SGEMM_VARIANT_TC05:
            return p.copy(split_k=split, stages=4, k_unroll=1)
    raise AssertionError("no tcgen05 plan compiled")


@pytest.mark.parametrize("split", [1, 4])
def test_stalled_kernel_reports_and_context_survives(split):
    M, N, K = 2, 2048, 1024
    x = synth.normal_bf16((M, K), 1.0, seed=1)
    W = synth.normal_bf16((N, K), 0.02, seed=2)
    xd, Wd = x.cuda(), W.cuda()
    plan = _tc05(split)
    sk.sgemm_device_errors()  # clear anything left over
    assert sk.sgemm_device_errors() == 0
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    sk.sgemm_bf16_skinny_ex(xd, Wd, y, plan=plan, flags=sk.SGEMM_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30, "bounded waits must end"
    assert torch.isnan(y.float()).all(), "outputs of a stalled kernel must be NaN"
    assert sk.sgemm_device_errors() & 1
    assert sk.sgemm_device_errors() == 0, "reading the error word clears it"
    # the context still works: the same call without the flag matches the oracle
    y2 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
    torch.cuda.synchronize()
    rep = compare(synth.bits(y2), oracle.skinny_gemm(synth.bits(x), synth.bits(W)),
                  synth.bits(x), synth.bits(W))
    assert rep["ok"], rep
    assert sk.sgemm_device_errors() == 0


def test_stalled_cluster_split_streaming_plan_reports_and_context_survives():
    """The cluster-split streaming plan's one wait (rank 0 for the other ranks'
    partial sums) runs out when they send none (the test-only flag): NaN
    outputs, the error bit, and a correct call afterwards."""
    M, N, K = 3, 2048, 4096
    x = synth.normal_bf16((M, K), 1.0, seed=11)
    W = synth.normal_bf16((N, K), 0.02, seed=12)
    xd, Wd = x.cuda(), W.cuda()
    base = next(p for p in (sk.sgemm_plan_get(i) for i in range(sk.sgemm_plan_count()))
                if p.variant == sk.SGEMM_VARIANT_LDG_CLUSTER)
    plan = base.copy(split_k=4)
    sk.sgemm_device_errors()
    assert sk.sgemm_device_errors() == 0
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    sk.sgemm_bf16_skinny_ex(xd, Wd, y, plan=plan, flags=sk.SGEMM_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30, "bounded waits must end"
    assert torch.isnan(y.float()).all(), "outputs of a stalled reduction must be NaN"
    assert sk.sgemm_device_errors() & 1
    assert sk.sgemm_device_errors() == 0
    y2 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
    torch.cuda.synchronize()
    rep = compare(synth.bits(y2), oracle.skinny_gemm(synth.bits(x), synth.bits(W)),
                  synth.bits(x), synth.bits(W))
    assert rep["ok"], rep
    assert sk.sgemm_device_errors() == 0
