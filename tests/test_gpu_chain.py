"""GPU: the elementwise step between GEMMs and a decode-step chain.

The chain follows the decode-chain workload (distinct weights per call, in the
order (12576,4096), (4096,4096), (2048,4096), (4096,1024), (8192,1536),
(4096,8192), (77440,4096), each output rescaled into the next input), shortened
to two calls per shape.  It runs as one CUDA graph with programmatic dependent
launch.  Each GEMM is checked against the oracle fed the GPU's actual input to
that GEMM, so errors do not compound, and each elementwise step is checked
bitwise against the same arithmetic on the CPU.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
import oracle
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare

pytestmark = pytest.mark.gpu

CHAIN_SHAPES = [(12576, 4096), (4096, 4096), (2048, 4096), (4096, 1024), (8192, 1536),
                (4096, 8192), (77440, 4096)]


def _rescale_cpu(y: torch.Tensor, n_dst: int, scale: float) -> torch.Tensor:
    yf = y.detach().cpu().float().reshape(-1)
    idx = torch.arange(n_dst) % yf.numel()
    return (yf[idx] * torch.tensor(scale, dtype=torch.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("n_src,n_dst", [(4096, 1536), (2048, 4096), (7, 100), (12576, 4096)])
def test_rescale_matches_cpu_bitwise(n_src, n_dst):
    y = synth.normal_bf16((1, n_src), 1.3, seed=n_src).cuda()
    x = torch.empty((1, n_dst), dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / (0.02 * math.sqrt(n_src))
    sk.sgemm_bf16_rescale(y, x, scale)
    torch.cuda.synchronize()
    ref = _rescale_cpu(y, n_dst, scale)
    assert torch.equal(x.cpu().reshape(-1).view(torch.int16), ref.view(torch.int16))


def test_rescale_rejects_bad_arguments():
    y = torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda")
    assert sk.load().sgemm_bf16_rescale(None, 8, y.data_ptr(), 8, 1.0, 0, None) == \
        sk.SGEMM_ERR_INVALID_ARG
    assert sk.load().sgemm_bf16_rescale(y.data_ptr(), 0, y.data_ptr(), 8, 1.0, 0, None) == \
        sk.SGEMM_ERR_INVALID_ARG
    assert sk.load().sgemm_bf16_rescale(y.data_ptr(), 8, y.data_ptr(), 8, 1.0, 16, None) == \
        sk.SGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("flags", [0, sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY])
def test_decode_chain_graph_per_gemm_parity(flags):
    seq = [s for s in CHAIN_SHAPES for _ in range(2)]
    Ws = [synth.normal_bf16(s, synth.W_STD, seed=50 + i, device="cuda") for i, s in enumerate(seq)]
    xs = [torch.empty((1, K), dtype=torch.bfloat16, device="cuda") for (_, K) in seq]
    ys = [torch.empty((1, N), dtype=torch.bfloat16, device="cuda") for (N, _) in seq]
    xs[0].copy_(synth.normal_bf16((1, seq[0][1]), 1.0, seed=49, device="cuda"))
    scales = [1.0 / (synth.W_STD * math.sqrt(K)) for (_, K) in seq]

    def step():
        for i in range(len(seq)):
            sk.sgemm_bf16_skinny_ex(xs[i], Ws[i], ys[i], flags=flags)
            if i + 1 < len(seq):
                sk.sgemm_bf16_rescale(ys[i], xs[i + 1], scales[i], flags=flags & sk.SGEMM_FLAG_PDL)

    step()
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for y in ys:
        y.zero_()
    g.replay()
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    for i, (N, K) in enumerate(seq):
        assert torch.equal(ys[i].view(torch.int16), eager[i].view(torch.int16)), i
        if i + 1 < len(seq):
            ref = _rescale_cpu(ys[i], seq[i + 1][1], scales[i])
            assert torch.equal(xs[i + 1].cpu().reshape(-1).view(torch.int16),
                               ref.view(torch.int16)), i
        rows = np.unique(np.concatenate([rng.choice(N, 48, replace=False), [0, N - 1]]))
        xb = synth.bits(xs[i])
        Wb = synth.bits(Ws[i][torch.as_tensor(rows, device="cuda")])
        rep = compare(synth.bits(ys[i])[:, rows], oracle.skinny_gemm(xb, Wb), xb, Wb)
        assert rep["ok"], (i, N, K, rep)
