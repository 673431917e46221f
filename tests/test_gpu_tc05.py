"""GPU parity of the TMA + tcgen05 kernel (SGEMM_VARIANT_TC05) against the oracle.

The kernel streams W with cp.async.bulk.tensor into a shared-memory ring and
multiplies on the 5th-generation tensor core with the accumulator in tensor
memory.  Its plans differ in ring depth, boxes per stage, the persistent
grid's CTAs per SM and the K split across a thread-block cluster (reduced in
distributed shared memory).  Each test runs the plans through the public C ABI
and compares with the CPU oracle (``tolerance.compare``), or checks bitwise
properties the design promises: the bits depend on (K, split) only.

Ordered small first: the first test is one CTA on one 64-element box.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
import oracle
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare

pytestmark = pytest.mark.gpu

DEV = "cuda"


def tc05(split=1, ring=4, nb=1, ctas=0):
    """A TC05 plan (threads 192, 128-row tiles)."""
    base = None
    for i in range(sk.sgemm_plan_count()):
        p = sk.sgemm_plan_get(i)
        if p.variant == sk.SGEMM_VARIANT_TC05:
            base = p
            break
    assert base is not None, "no TC05 kernel compiled"
    return base.copy(split_k=split, stages=ring, k_unroll=nb, ctas_per_sm=ctas)


def _inputs(M, N, K, seed, fam="normal", wstd=synth.W_STD):
    x = synth.family_bf16((M, K), fam, synth.X_STD, seed=seed)
    W = synth.family_bf16((N, K), fam, wstd, seed=seed + 1)
    return x, W


def _check(x, W, y, rows=None):
    xb, Wb, yb = synth.bits(x), synth.bits(W), synth.bits(y)
    if rows is not None:
        Wb = Wb[rows]
        yb = yb[:, rows]
    rep = compare(yb, oracle.skinny_gemm(xb, Wb), xb, Wb)
    assert rep["ok"], rep
    return rep


def _run(x, W, plan, **kw):
    y = sk.sgemm_bf16_skinny_ex(x.to(DEV), W.to(DEV), plan=plan, **kw)
    torch.cuda.synchronize()
    return y


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sk.load()
    yield
    assert sk.sgemm_device_errors() == 0


# ---------------------------------------------------------------- one CTA first
@pytest.mark.parametrize("M", [1, 4, 8])
def test_one_tile_one_box(M):
    x, W = _inputs(M, 128, 64, seed=1)
    _check(x, W, _run(x, W, tc05(ring=2)))


@pytest.mark.parametrize("N,K", [(1, 8), (5, 40), (129, 72), (200, 128), (613, 2600),
                                 (1000, 1536), (2049, 256), (64, 8200)])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_ragged_shapes(M, N, K):
    x, W = _inputs(M, N, K, seed=N + K)
    _check(x, W, _run(x, W, tc05()))


# ------------------------------------------------------------ plan geometry
@pytest.mark.parametrize("split", [1, 2, 3, 5, 8, 16])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_cluster_splits(M, split):
    """Every M: the other ranks push rows of M partial sums with 16-byte (M = 4, 8),
    8-byte (M = 2, 6) or 4-byte (odd M) stores into rank 0."""
    N, K = 613, 2600  # 41 boxes of K: ragged last box, splits of 21/14/9/6/3 boxes
    x, W = _inputs(M, N, K, seed=20 + split)
    y = _run(x, W, tc05(split=split))
    _check(x, W, y)


@pytest.mark.parametrize("ring,nb", [(2, 1), (3, 1), (8, 1), (12, 1), (2, 2), (4, 2), (6, 2),
                                     (2, 3), (4, 3), (2, 4), (3, 4)])
def test_ring_and_boxes_per_stage_do_not_change_bits(ring, nb):
    M, N, K = 3, 1500, 3072
    x, W = _inputs(M, N, K, seed=30)
    for split in (1, 3):
        ref = _run(x, W, tc05(split=split, ring=4, nb=1))
        y = _run(x, W, tc05(split=split, ring=ring, nb=nb))
        assert torch.equal(ref.view(torch.int16), y.view(torch.int16)), (split, ring, nb)
    _check(x, W, y)


@pytest.mark.parametrize("ctas", [1, 2, 3])
def test_persistent_grid_sizes(ctas):
    """Fewer CTAs than tiles: each CTA walks several tiles through the two
    alternating accumulators; the bits do not depend on the grid."""
    M, N, K = 2, 77440 // 4, 1024  # 152 tiles
    x, W = _inputs(M, N, K, seed=40)
    ref = _run(x, W, tc05())
    y = _run(x, W, tc05(ctas=ctas))
    assert torch.equal(ref.view(torch.int16), y.view(torch.int16))
    _check(x, W, y)


def test_deterministic_and_m_independent():
    N, K = 4096, 4096
    x, W = _inputs(8, N, K, seed=50)
    xd, Wd = x.to(DEV), W.to(DEV)
    for plan in (tc05(), tc05(split=4), tc05(split=8, ring=3, nb=2)):
        y8 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
        y8b = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
        torch.cuda.synchronize()
        assert torch.equal(y8.view(torch.int16), y8b.view(torch.int16)), plan
        for m in range(8):
            y1 = sk.sgemm_bf16_skinny_ex(xd[m:m + 1], Wd, plan=plan)
            torch.cuda.synchronize()
            assert torch.equal(y1.view(torch.int16)[0], y8.view(torch.int16)[m]), (plan, m)
        _check(x, W, y8)


@pytest.mark.parametrize("fam", synth.FAMILIES)
def test_input_families(fam):
    x, W = _inputs(4, 611, 2048, seed=60, fam=fam)
    for split in (1, 4):
        _check(x, W, _run(x, W, tc05(split=split)))


# ------------------------------------------------------------ full-size shapes
def _sample_rows(N, n=96, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=min(n, N), replace=False).tolist()) | {0, 1, N - 2, N - 1}
    return np.array(sorted(rows))


@pytest.mark.parametrize("N,K,split", [(12576, 4096, 1), (12576, 4096, 3), (4096, 4096, 8),
                                       (2048, 4096, 16), (4096, 1024, 4), (8192, 1536, 2),
                                       (4096, 8192, 8), (77440, 4096, 1)])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_full_size_shapes_sampled(M, N, K, split):
    xd = synth.normal_bf16((M, K), synth.X_STD, seed=100 + M, device=DEV)
    Wd = synth.normal_bf16((N, K), synth.W_STD, seed=200, device=DEV)
    y = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=tc05(split=split))
    torch.cuda.synchronize()
    rows = _sample_rows(N, seed=N)
    x = xd.cpu()
    Ws = Wd[torch.as_tensor(rows, device=DEV)].cpu()
    rep = compare(synth.bits(y)[:, rows], oracle.skinny_gemm(synth.bits(x), synth.bits(Ws)),
                  synth.bits(x), synth.bits(Ws))
    assert rep["ok"], rep


# -------------------------------------------------------- layouts and epilogues
def test_strided_x_and_y_and_guard_bands():
    M, N, K = 3, 999, 1024
    x, W = _inputs(M, N, K, seed=70)
    big = torch.zeros((M, K + 64), dtype=torch.bfloat16, device=DEV)
    big[:, 8:8 + K] = x.to(DEV)
    xv = big[:, 8:8 + K]
    ybig = torch.full((M, N + 13), 7.0, dtype=torch.bfloat16, device=DEV)
    for split in (1, 2):
        sk.sgemm_bf16_skinny_ex(xv, W.to(DEV), ybig[:, :N], plan=tc05(split=split))
        torch.cuda.synchronize()
        _check(x, W, ybig[:, :N].contiguous())
        assert torch.all(ybig[:, N:] == 7.0), "wrote outside y"


@pytest.mark.parametrize("batch", [2, 8])
@pytest.mark.parametrize("split", [1, 2])
def test_batched_matches_separate_calls(batch, split):
    M, N, K = 3, 4096, 128
    act = synth.normal_bf16((M, batch * K), 1.0, seed=80 + batch).to(DEV)
    xs = act.unflatten(1, (batch, K)).transpose(0, 1)  # strided views, row stride batch*K
    Ws = [synth.normal_bf16((N, K), synth.PAIR_W_STD, seed=90 + i).to(DEV) for i in range(batch)]
    plan = tc05(split=split)
    outs = sk.sgemm_bf16_skinny_batched_ex([(xs[i], Ws[i]) for i in range(batch)], plan=plan)
    torch.cuda.synchronize()
    for i in range(batch):
        sep = sk.sgemm_bf16_skinny_ex(xs[i], Ws[i], plan=plan)
        torch.cuda.synchronize()
        assert torch.equal(sep.view(torch.int16), outs[i].view(torch.int16))
        _check(xs[i].contiguous().cpu(), Ws[i].cpu(), outs[i])


@pytest.mark.parametrize("split", [1, 4])
def test_fp32_output_and_fused_chain_step(split):
    from tolerance import compare_f32
    M, N, K = 4, 1111, 2048
    x, W = _inputs(M, N, K, seed=100)
    xd, Wd = x.to(DEV), W.to(DEV)
    plan = tc05(split=split)
    y = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
    y32 = sk.sgemm_bf16_skinny_f32out_ex(xd, Wd, plan=plan)
    yc = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    xn = torch.empty((M, 3000), dtype=torch.bfloat16, device=DEV)
    sk.sgemm_bf16_skinny_rescale_ex(xd, Wd, yc, xn, 0.375, plan=plan)
    torch.cuda.synchronize()
    r = compare_f32(y32.cpu().view(torch.int32).numpy().view(np.uint32),
                    oracle.skinny_gemm_f32(synth.bits(x), synth.bits(W)), synth.bits(x), synth.bits(W))
    assert r["ok"], r
    # rounding the FP32 sums gives the BF16 outputs; the fused step changes nothing in y
    assert torch.equal(y32.to(torch.bfloat16).view(torch.int16), y.view(torch.int16))
    assert torch.equal(yc.view(torch.int16), y.view(torch.int16))
    want = (yc.cpu().float()[:, torch.arange(3000) % N] * 0.375).to(torch.bfloat16)
    assert torch.equal(xn.cpu().view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("flags", [sk.SGEMM_FLAG_PDL,
                                   sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY])
def test_pdl_chain_matches_plain_launches_and_graph(flags):
    M = 2
    shapes = [(4096, 4096), (12576, 4096), (2048, 4096), (4096, 2048)]
    Ws = [synth.normal_bf16(s, synth.W_STD, seed=110 + i).to(DEV) for i, s in enumerate(shapes)]
    x0 = synth.normal_bf16((M, 4096), 1.0, seed=109).to(DEV)
    plans = [tc05(split=4), tc05(), tc05(split=8), tc05(split=2, ring=3, nb=2)]

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
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gout = chain(flags)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, gout):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_graph_replay_sees_in_place_weight_refresh():
    M, N, K = 2, 2048, 4096
    x, W = _inputs(M, N, K, seed=120)
    xd, Wd = x.to(DEV), W.to(DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    plan = tc05(split=4)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sk.sgemm_bf16_skinny_ex(xd, Wd, y, plan=plan)
    g.replay()
    torch.cuda.synchronize()
    _check(x, W, y)
    W2 = synth.normal_bf16((N, K), synth.W_STD, seed=121)
    Wd.copy_(W2.to(DEV))
    g.replay()
    torch.cuda.synchronize()
    _check(x, W2, y)


# ------------------------------------------------------------- plan checks
def test_plan_checks():
    ok = tc05()
    assert sk.sgemm_plan_check(ok, 1, 4096, 4096) == sk.SGEMM_OK
    bad = [ok.copy(threads=128), ok.copy(k_unroll=5), ok.copy(stages=1), ok.copy(stages=17),
           ok.copy(split_k=17), ok.copy(lanes_per_row=4), ok.copy(rows_per_warp=64),
           ok.copy(stages=16, k_unroll=4)]  # 16 x 4 boxes x 18 KiB do not fit shared memory
    for p in bad:
        assert sk.sgemm_plan_check(p, 1, 4096, 4096) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE, p
    # more splits than 64-element boxes of K
    assert sk.sgemm_plan_check(ok.copy(split_k=2), 1, 16, 64) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE
    assert sk.sgemm_plan_check(ok.copy(split_k=2), 1, 16, 72) == sk.SGEMM_OK
