"""GPU: the two epilogue forms of the GEMM.

1. FP32 outputs (``sgemm_bf16_skinny_f32out_ex``): every plan against the
   oracle's exact sum rounded once to FP32, on the router-gate shape (288, 4096)
   that vLLM PR #62949 (Validation, the nsys census) leaves on cuBLAS for its
   FP32 output, and on a ragged shape.  Since only the store differs, the BF16
   rounding of the FP32 output must equal that plan's BF16 output bitwise.
2. The decode chain's elementwise step fused into the epilogue
   (``sgemm_bf16_skinny_rescale_ex``): y bitwise equal to the plain call, and
   the next input bitwise equal to the same step done on the CPU from y (which
   is what ``sgemm_bf16_rescale`` computes), including wrap-around
   (n_next > N), strided rows and a PDL chain under graph capture.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
import oracle
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare, compare_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _all_plans():
    sk.load()
    return [sk.sgemm_plan_get(i) for i in range(sk.sgemm_plan_count())]


def _inputs(M, N, K, seed):
    x = synth.normal_bf16((M, K), synth.X_STD, seed=seed)
    W = synth.normal_bf16((N, K), synth.W_STD, seed=seed + 1)
    return x, W


def _f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


# ------------------------------------------------------------------ FP32 out
@pytest.mark.parametrize("N,K", [(288, 4096), (613, 2600)])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_f32_output_every_plan(M, N, K):
    x, W = _inputs(M, N, K, seed=3100 + N + M)
    xd, Wd = x.to(DEV), W.to(DEV)
    xb, Wb = synth.bits(x), synth.bits(W)
    ref = oracle.skinny_gemm_f32(xb, Wb)
    for p in _all_plans():
        for split in (1, 2):
            plan = p.copy(split_k=split)
            if sk.sgemm_plan_check(plan, M, N, K) != sk.SGEMM_OK:
                continue
            y32 = sk.sgemm_bf16_skinny_f32out_ex(xd, Wd, plan=plan)
            y16 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
            torch.cuda.synchronize()
            rep = compare_f32(_f32_bits(y32), ref, xb, Wb)
            assert rep["ok"], (plan, rep)
            # the same sums: rounding them to BF16 gives the BF16 output exactly
            assert torch.equal(y32.to(torch.bfloat16).view(torch.int16),
                               y16.view(torch.int16)), plan


def test_f32_output_strided_and_graph():
    M, N, K = 4, 288, 4096
    x, W = _inputs(M, N, K, seed=3200)
    xd, Wd = x.to(DEV), W.to(DEV)
    big = torch.full((M, N + 40), -7.0, dtype=torch.float32, device=DEV)
    yv = big[:, 8:8 + N]
    sk.sgemm_bf16_skinny_f32out_ex(xd, Wd, yv)
    torch.cuda.synchronize()
    eager = yv.clone()
    assert torch.all(big[:, :8] == -7.0) and torch.all(big[:, 8 + N:] == -7.0)
    rep = compare_f32(_f32_bits(eager), oracle.skinny_gemm_f32(synth.bits(x), synth.bits(W)),
                      synth.bits(x), synth.bits(W))
    assert rep["ok"], rep
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sk.sgemm_bf16_skinny_f32out_ex(xd, Wd, yv,
                                          flags=sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY)
    torch.cuda.current_stream().wait_stream(s)
    yv.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(yv.view(torch.int32), eager.view(torch.int32))


def test_f32_output_rejects_misaligned_y():
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    buf = torch.zeros(40, dtype=torch.float32, device=DEV)
    st = sk.load().sgemm_bf16_skinny_f32out_ex(x.data_ptr(), 64, W.data_ptr(),
                                               buf.data_ptr() + 2, 16, 1, 16, 64, None, 0, None)
    assert st == sk.SGEMM_ERR_MISALIGNED


# --------------------------------------------------------- fused chain step
def _rescale_cpu(y: torch.Tensor, n_next: int, scale: float) -> torch.Tensor:
    """x_next[m, k] = bf16(float(y[m, k mod N]) * scale), FP32 multiply, RNE."""
    yf = y.detach().cpu().float()
    idx = torch.arange(n_next) % yf.shape[1]
    return (yf[:, idx] * torch.tensor(scale, dtype=torch.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("N,K,n_next", [(613, 2600, 1536), (613, 2600, 613), (613, 2600, 2000),
                                        (4096, 1024, 4096), (2048, 4096, 8192)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_fused_rescale_every_plan(M, N, K, n_next):
    x, W = _inputs(M, N, K, seed=3300 + N + n_next)
    xd, Wd = x.to(DEV), W.to(DEV)
    scale = 1.0 / (synth.W_STD * math.sqrt(K))
    seen = 0
    for p, split in ((p, s) for p in _all_plans() for s in (1, 2)):
        plan = p.copy(split_k=split)
        if sk.sgemm_plan_check(plan, M, N, K) != sk.SGEMM_OK:
            continue
        y_plain = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        xn = torch.full((M, n_next), 3.0, dtype=torch.bfloat16, device=DEV)
        sk.sgemm_bf16_skinny_rescale_ex(xd, Wd, y, xn, scale, plan=plan)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_plain.view(torch.int16)), plan
        ref = _rescale_cpu(y, n_next, scale)
        assert torch.equal(xn.cpu().view(torch.int16), ref.view(torch.int16)), plan
        seen += 1
    assert seen > 20
    rep = compare(synth.bits(y_plain), oracle.skinny_gemm(synth.bits(x), synth.bits(W)),
                  synth.bits(x), synth.bits(W))
    assert rep["ok"], rep


def test_fused_rescale_strided_rows_leave_gaps_alone():
    M, N, K, n_next = 2, 1000, 1024, 1536
    x, W = _inputs(M, N, K, seed=3400)
    big = torch.full((M, n_next + 24), 5.0, dtype=torch.bfloat16, device=DEV)
    xn = big[:, 8:8 + n_next]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sk.sgemm_bf16_skinny_rescale_ex(x.to(DEV), W.to(DEV), y, xn, 0.25)
    torch.cuda.synchronize()
    assert torch.all(big[:, :8] == 5.0) and torch.all(big[:, 8 + n_next:] == 5.0)
    assert torch.equal(xn.cpu().view(torch.int16), _rescale_cpu(y, n_next, 0.25).view(torch.int16))


def test_fused_rescale_rejects_overlap():
    x = torch.zeros((1, 1024), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((512, 1024), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((1, 512), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sk.SgemmError):
        sk.sgemm_bf16_skinny_rescale_ex(x, W, y, x, 1.0)        # x_next is x
    with pytest.raises(sk.SgemmError):
        sk.sgemm_bf16_skinny_rescale_ex(x, W, y, y, 1.0)        # x_next is y


CHAIN_SHAPES = [(12576, 4096), (4096, 4096), (2048, 4096), (4096, 1024), (8192, 1536),
                (4096, 8192), (77440, 4096)]


@pytest.mark.parametrize("flags", [0, sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY])
def test_fused_decode_chain_equals_separate_steps(flags):
    """The decode-chain workload (two GEMMs per shape here) with the elementwise
    step fused, eager and replayed from a CUDA graph, against the same chain with
    the separate elementwise kernel: every y and every x bitwise equal."""
    seq = [s for s in CHAIN_SHAPES for _ in range(2)]
    Ws = [synth.normal_bf16(s, synth.W_STD, seed=3500 + i, device=DEV) for i, s in enumerate(seq)]
    x0 = synth.normal_bf16((1, seq[0][1]), 1.0, seed=3499, device=DEV)
    scales = [1.0 / (synth.W_STD * math.sqrt(K)) for (_, K) in seq]

    def buffers():
        xs = [torch.empty((1, K), dtype=torch.bfloat16, device=DEV) for (_, K) in seq]
        ys = [torch.empty((1, N), dtype=torch.bfloat16, device=DEV) for (N, _) in seq]
        xs[0].copy_(x0)
        return xs, ys

    xs_a, ys_a = buffers()
    for i in range(len(seq)):
        sk.sgemm_bf16_skinny_ex(xs_a[i], Ws[i], ys_a[i], flags=flags)
        if i + 1 < len(seq):
            sk.sgemm_bf16_rescale(ys_a[i], xs_a[i + 1], scales[i], flags=flags & sk.SGEMM_FLAG_PDL)
    xs_b, ys_b = buffers()

    def fused():
        for i in range(len(seq)):
            if i + 1 < len(seq):
                sk.sgemm_bf16_skinny_rescale_ex(xs_b[i], Ws[i], ys_b[i], xs_b[i + 1], scales[i],
                                                flags=flags)
            else:
                sk.sgemm_bf16_skinny_ex(xs_b[i], Ws[i], ys_b[i], flags=flags)

    fused()
    torch.cuda.synchronize()
    for i in range(len(seq)):
        assert torch.equal(ys_a[i].view(torch.int16), ys_b[i].view(torch.int16)), i
        assert torch.equal(xs_a[i].view(torch.int16), xs_b[i].view(torch.int16)), i
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fused()
    torch.cuda.current_stream().wait_stream(s)
    for t in ys_b + xs_b[1:]:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for i in range(len(seq)):
        assert torch.equal(ys_a[i].view(torch.int16), ys_b[i].view(torch.int16)), i
        assert torch.equal(xs_a[i].view(torch.int16), xs_b[i].view(torch.int16)), i


# ------------------------------------------------------ merged projections
def test_two_projections_of_one_input_in_one_launch():
    """Two projections of the same x (the f_a/g_a merge of lmdeploy PR #4968,
    "feat(pytorch): add glm5.3-flash support", Optimizations: merging them cuts
    the KDA projection launches) in one batched launch, sharing the x buffer,
    and as one GEMM over the stacked weight [W_a; W_b] with the same plan: both
    equal the separate calls bitwise."""
    M, K = 2, 2048
    Na, Nb = 768, 1280
    x = synth.normal_bf16((M, K), synth.X_STD, seed=3600).to(DEV)
    Wa = synth.normal_bf16((Na, K), synth.W_STD, seed=3601).to(DEV)
    Wb = synth.normal_bf16((Na, K), synth.W_STD, seed=3602).to(DEV)
    plan = sk.sgemm_plan_select(Na, K, M)
    ya, yb = sk.sgemm_bf16_skinny_batched_ex([(x, Wa), (x, Wb)], plan=plan)
    sa = sk.sgemm_bf16_skinny_ex(x, Wa, plan=plan)
    sb = sk.sgemm_bf16_skinny_ex(x, Wb, plan=plan)
    torch.cuda.synchronize()
    assert torch.equal(ya.view(torch.int16), sa.view(torch.int16))
    assert torch.equal(yb.view(torch.int16), sb.view(torch.int16))
    # unequal widths: one GEMM over the stacked weight; a CUDA-core plan's order
    # per output depends only on K and its lanes per row, not on N
    Wc = synth.normal_bf16((Nb, K), synth.W_STD, seed=3603).to(DEV)
    stacked = torch.cat([Wa, Wc], 0)
    plan = sk.sgemm_plan_select(Na + Nb, K, M).copy(variant=sk.SGEMM_VARIANT_LDG_MIXFMA,
                                                     rows_per_warp=1, lanes_per_row=32,
                                                     k_unroll=8, split_k=1, stages=1)
    y = sk.sgemm_bf16_skinny_ex(x, stacked, plan=plan)
    sa = sk.sgemm_bf16_skinny_ex(x, Wa, plan=plan)
    sc = sk.sgemm_bf16_skinny_ex(x, Wc, plan=plan)
    torch.cuda.synchronize()
    assert torch.equal(y[:, :Na].view(torch.int16), sa.view(torch.int16))
    assert torch.equal(y[:, Na:].view(torch.int16), sc.view(torch.int16))
    xb = synth.bits(x.cpu())
    rep = compare(synth.bits(y), oracle.skinny_gemm(xb, synth.bits(stacked.cpu())), xb,
                  synth.bits(stacked.cpu()))
    assert rep["ok"], rep
