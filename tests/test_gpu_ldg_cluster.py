"""GPU parity of the cluster-split streaming plans (SGEMM_VARIANT_LDG_CLUSTER).

These run the mixed-precision streaming kernels with their K split across a
thread-block cluster: rank 0 takes the other ranks' FP32 partial sums into its
shared memory and adds them in split order from 0, as the second-pass kernel of
variant 1 does.  So each output is checked against the oracle and bitwise
against variant 1 with the same split (two launches, scratch memory).
"""
from __future__ import annotations

import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
import oracle
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _cl_plans():
    """The compiled cluster-split plans (one per configuration and CTA size)."""
    return [p for p in (sk.sgemm_plan_get(i) for i in range(sk.sgemm_plan_count()))
            if p.variant == sk.SGEMM_VARIANT_LDG_CLUSTER]


def _two_kernel(p):
    """The same configuration as a variant-1 plan: scratch split plus second pass."""
    return p.copy(variant=sk.SGEMM_VARIANT_LDG_MIXFMA)


def _inputs(M, N, K, seed):
    x = synth.normal_bf16((M, K), synth.X_STD, seed=seed)
    W = synth.normal_bf16((N, K), synth.W_STD, seed=seed + 1)
    return x, W


def _eq(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sk.load()
    sk.sgemm_init()
    yield
    assert sk.sgemm_device_errors() == 0


@pytest.mark.parametrize("split", [2, 3, 5, 8])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_every_kernel_matches_two_kernel_split(M, split):
    N, K = 613, 2600  # ragged rows and a ragged last split
    x, W = _inputs(M, N, K, seed=500 + M)
    xd, Wd = x.to(DEV), W.to(DEV)
    xb, Wb = synth.bits(x), synth.bits(W)
    ref = oracle.skinny_gemm(xb, Wb)
    plans = _cl_plans()
    assert plans
    for p in plans:
        one = p.copy(split_k=split)
        two = _two_kernel(one)
        assert sk.sgemm_plan_check(one, M, N, K) == sk.SGEMM_OK, one
        y1 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=one)
        y2 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=two)
        torch.cuda.synchronize()
        assert _eq(y1, y2), one
        rep = compare(synth.bits(y1), ref, xb, Wb)
        assert rep["ok"], (one, rep)


@pytest.mark.parametrize("N,K", [(1, 16), (7, 64), (300, 1000), (2048, 4096), (8192, 1536),
                                 (4096, 1024)])
@pytest.mark.parametrize("M", [1, 4])
def test_shapes(M, N, K):
    x, W = _inputs(M, N, K, seed=600 + N)
    xd, Wd = x.to(DEV), W.to(DEV)
    for p in _cl_plans()[:4]:
        for split in (2, 4):
            one = p.copy(split_k=split)
            if sk.sgemm_plan_check(one, M, N, K) != sk.SGEMM_OK:
                assert K < 8 * 2 * split, (one, N, K)  # too few 8-element chunks to split
                continue
            y = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=one)
            y2 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=_two_kernel(one))
            torch.cuda.synchronize()
            assert _eq(y, y2), one
            if N * K <= 4096 * 1024:
                rep = compare(synth.bits(y), oracle.skinny_gemm(synth.bits(x), synth.bits(W)),
                              synth.bits(x), synth.bits(W))
                assert rep["ok"], rep


def test_strided_batched_and_epilogues():
    from tolerance import compare_f32
    M, N, K, batch = 3, 1111, 2048, 3
    one = _cl_plans()[0].copy(split_k=4)
    act = synth.normal_bf16((M, batch * K), 1.0, seed=700).to(DEV)
    xs = act.unflatten(1, (batch, K)).transpose(0, 1)
    Ws = [synth.normal_bf16((N, K), synth.W_STD, seed=701 + i).to(DEV) for i in range(batch)]
    outs = sk.sgemm_bf16_skinny_batched_ex([(xs[i], Ws[i]) for i in range(batch)], plan=one)
    y32 = sk.sgemm_bf16_skinny_f32out_ex(xs[0], Ws[0], plan=one)
    yc = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    xn = torch.empty((M, 3000), dtype=torch.bfloat16, device=DEV)
    sk.sgemm_bf16_skinny_rescale_ex(xs[0], Ws[0], yc, xn, 0.375, plan=one)
    torch.cuda.synchronize()
    for i in range(batch):
        sep = sk.sgemm_bf16_skinny_ex(xs[i], Ws[i], plan=one)
        torch.cuda.synchronize()
        assert _eq(sep, outs[i])
        xb, Wb = synth.bits(xs[i].contiguous().cpu()), synth.bits(Ws[i].cpu())
        rep = compare(synth.bits(outs[i]), oracle.skinny_gemm(xb, Wb), xb, Wb)
        assert rep["ok"], rep
    xb, Wb = synth.bits(xs[0].contiguous().cpu()), synth.bits(Ws[0].cpu())
    r = compare_f32(y32.cpu().view(torch.int32).numpy().view("uint32"),
                    oracle.skinny_gemm_f32(xb, Wb), xb, Wb)
    assert r["ok"], r
    assert _eq(y32.to(torch.bfloat16), outs[0])
    assert _eq(yc, outs[0])
    want = (yc.cpu().float()[:, torch.arange(3000) % N] * 0.375).to(torch.bfloat16)
    assert _eq(xn.cpu(), want)


@pytest.mark.parametrize("flags", [sk.SGEMM_FLAG_PDL,
                                   sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY])
def test_pdl_chain_and_graph(flags):
    M = 2
    shapes = [(4096, 4096), (2048, 4096), (4096, 2048), (8192, 4096)]  # N_i >= K_{i+1}
    Ws = [synth.normal_bf16(s, synth.W_STD, seed=800 + i).to(DEV) for i, s in enumerate(shapes)]
    x0 = synth.normal_bf16((M, 4096), 1.0, seed=799).to(DEV)
    base = _cl_plans()[0]
    plans = [base.copy(split_k=s) for s in (4, 2, 3, 8)]

    def chain(fl):
        outs, x = [], x0
        for i, W in enumerate(Ws):
            y = torch.empty((M, W.shape[0]), dtype=torch.bfloat16, device=DEV)
            sk.sgemm_bf16_skinny_ex(x, W, y, plan=plans[i], flags=fl)
            outs.append(y)
            if i + 1 < len(Ws):
                x = (y[:, :Ws[i + 1].shape[1]].float() * 8.0).to(torch.bfloat16)
        return outs

    ref = chain(0)
    torch.cuda.synchronize()
    got = chain(flags)
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert _eq(a, b)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gout = chain(flags)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ref, gout):
            assert _eq(a, b)
