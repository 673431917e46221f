"""Failure detection on the GPU, without a GPU fault.

The bulk-copy kernel waits on shared-memory mbarriers for its data.  Every
wait is bounded (about 0.2 s); when one gives up, the kernel writes NaN to the
outputs it owns, sets the device error word and returns, so the context stays
usable.  The test-only launch flag SGEMM_FLAG_TEST_STALL makes the kernel's
producer issue no copies at all, so the waits run out: nothing faults, traps or
hangs.  The host reads the status with sgemm_device_errors().
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
from bf16_skinny_gemm_gb300 import synth

pytestmark = pytest.mark.gpu


def _bulk_plan():
    for i in range(sk.sgemm_plan_count()):
        p = sk.sgemm_plan_get(i)
        if p.variant == sk.SGEMM_VARIANT_BULK:
            return p
    raise AssertionError("no bulk plan compiled")


def test_stalled_bulk_kernel_reports_and_context_survives():
    M, N, K = 2, 2048, 1024
    x = synth.normal_bf16((M, K), 1.0, seed=1).cuda()
    W = synth.normal_bf16((N, K), 0.02, seed=2).cuda()
    plan = _bulk_plan()
    assert sk.sgemm_device_errors() in (0, 1)  # clear anything left over
    assert sk.sgemm_device_errors() == 0
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    sk.sgemm_bf16_skinny_ex(x, W, y, plan=plan, flags=sk.SGEMM_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert elapsed < 30, "bounded waits must end"
    assert torch.isnan(y.float()).all(), "outputs of a stalled kernel must be NaN"
    assert sk.sgemm_device_errors() & 1
    assert sk.sgemm_device_errors() == 0, "reading the error word clears it"
    # the context still works: the same call without the flag is correct
    y2 = sk.sgemm_bf16_skinny_ex(x, W, plan=plan)
    ref = (x.double() @ W.double().T)
    torch.cuda.synchronize()
    err = (y2.double() - ref).abs().max().item()
    assert np.isfinite(err) and err < 0.05
    assert sk.sgemm_device_errors() == 0
