"""GPU parity: the CUDA library, called through its C ABI, against the CPU oracle.

Every comparison uses ``tolerance.compare``: the stated per-element bound
(2 BF16 ulp + 1e-3 sqrt(K) max|x| max|W|), the tighter bound derived from
FP32 accumulation, and cosine >= 0.99999 per output row; NaN / inf must match
in kind.  Shapes span several CTAs, every lane layout and ragged tails; the
full-size decode shapes are checked on sampled output rows, which the oracle
computes one by one.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_skinny_gemm_gb300 as sk
import golden_cases
import oracle
from bf16_skinny_gemm_gb300 import synth
from tolerance import compare

pytestmark = pytest.mark.gpu

DEV = "cuda"

SWEEP_SHAPES = [(12576, 4096), (4096, 4096), (2048, 4096), (4096, 1024), (8192, 1536),
                (4096, 8192)]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sk.load()
    sk.sgemm_init()
    yield


def _inputs(M, N, K, seed, fam="normal", wstd=synth.W_STD):
    x = synth.family_bf16((M, K), fam, synth.X_STD, seed=seed)
    W = synth.family_bf16((N, K), fam, wstd, seed=seed + 1)
    return x, W


def _check(x, W, y, rows=None, tight=True):
    xb, Wb = synth.bits(x), synth.bits(W)
    yb = synth.bits(y)
    if rows is not None:
        Wb = Wb[rows]
        yb = yb[:, rows]
    ref = oracle.skinny_gemm(xb, Wb)
    rep = compare(yb, ref, xb, Wb, tight=tight)
    assert rep["ok"], rep
    return rep


# ---------------------------------------------------------------- small shapes
SMALL = [(1, 8), (1, 64), (7, 264), (33, 128), (300, 1024), (1000, 1536), (517, 4096),
         (2049, 256), (64, 8200), (5, 40)]


@pytest.mark.parametrize("N,K", SMALL)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_small_shapes_default_plan(M, N, K):
    x, W = _inputs(M, N, K, seed=N * 7 + K)
    y = sk.sgemm_bf16_skinny(x.to(DEV), W.to(DEV))
    torch.cuda.synchronize()
    _check(x, W, y)


@pytest.mark.parametrize("fam", synth.FAMILIES)
@pytest.mark.parametrize("M", [1, 4, 8])
def test_input_families(fam, M):
    x, W = _inputs(M, 611, 2048, seed=5, fam=fam)
    y = sk.sgemm_bf16_skinny(x.to(DEV), W.to(DEV))
    torch.cuda.synchronize()
    _check(x, W, y)


def _all_plans():
    sk.load()
    return [sk.sgemm_plan_get(i) for i in range(sk.sgemm_plan_count())]


@pytest.mark.parametrize("split", [1, 2, 3, 5])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 6, 8])
def test_every_plan_every_split(M, split):
    N, K = 613, 2600
    x, W = _inputs(M, N, K, seed=11)
    xd, Wd = x.to(DEV), W.to(DEV)
    xb, Wb = synth.bits(x), synth.bits(W)
    ref = oracle.skinny_gemm(xb, Wb)
    for p in _all_plans():
        plan = p.copy(split_k=split)
        assert sk.sgemm_plan_check(plan, M, N, K) == sk.SGEMM_OK, plan
        y = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
        torch.cuda.synchronize()
        rep = compare(synth.bits(y), ref, xb, Wb)
        assert rep["ok"], (plan, rep)


@pytest.mark.parametrize("ctas", [1, 2, 5])
def test_grid_sizing_does_not_change_results(ctas):
    N, K, M = 2111, 1536, 2
    x, W = _inputs(M, N, K, seed=12)
    xd, Wd = x.to(DEV), W.to(DEV)
    base = sk.sgemm_plan_select(N, K, M)
    y0 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=base)
    y1 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=base.copy(ctas_per_sm=ctas))
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    _check(x, W, y1)


# ---------------------------------------------------------- golden closed forms
@pytest.mark.parametrize("case", golden_cases.load(), ids=lambda c: c.name)
def test_golden_cases_on_gpu(case):
    """Hand-derived cases, zero-padded to a multiple of 8 in K (zeros add exact
    zero products).  Cases whose FP32 evaluation is exact must match bitwise."""
    Kp = (case.K + 7) // 8 * 8
    x = np.zeros((case.M, Kp), np.uint16)
    W = np.zeros((case.N, Kp), np.uint16)
    x[:, :case.K] = case.x
    W[:, :case.K] = case.W
    y = sk.sgemm_bf16_skinny(synth.from_bits(x, DEV), synth.from_bits(W, DEV))
    torch.cuda.synchronize()
    yb = synth.bits(y)
    # 2^100 + 1 - 2^100: the 1 is below FP32 resolution next to 2^100, so no
    # FP32 accumulation keeps it; only the element bounds apply there
    y_ref = np.where(case.y_nan, np.uint16(0x7FC0), case.y).astype(np.uint16)
    rep = compare(yb, y_ref, x, W, cosine=case.name != "cancellation")
    nan = ((yb & 0x7F80) == 0x7F80) & ((yb & 0x7F) != 0)
    assert np.array_equal(nan, case.y_nan), case.name
    assert rep["ok"], (case.name, rep)
    exact_in_fp32 = case.name not in ("cancellation", "sticky_rounds_up", "subnormal_rounds_up",
                                      "max_plus_half_ulp", "max_plus_quarter_ulp")
    if exact_in_fp32:
        sel = ~case.y_nan
        assert np.array_equal(yb[sel], case.y[sel]), case.name


# ----------------------------------------------------------- properties
@pytest.mark.parametrize("MX", [4, 8])
def test_deterministic_and_m_independent(MX):
    N, K = 4096, 4096
    x, W = _inputs(MX, N, K, seed=13)
    xd, Wd = x.to(DEV), W.to(DEV)
    for p in _all_plans():
        y4 = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=p)
        y4b = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=p)
        torch.cuda.synchronize()
        assert torch.equal(y4.view(torch.int16), y4b.view(torch.int16)), p
        for m in range(MX):
            y1 = sk.sgemm_bf16_skinny_ex(xd[m:m + 1], Wd, plan=p)
            torch.cuda.synchronize()
            assert torch.equal(y1.view(torch.int16)[0], y4.view(torch.int16)[m]), (p, m)


def test_strided_x_and_y():
    M, N, K = 3, 999, 1024
    x, W = _inputs(M, N, K, seed=14)
    big = torch.zeros((M, K + 64), dtype=torch.bfloat16, device=DEV)
    big[:, 8:8 + K] = x.to(DEV)
    xv = big[:, 8:8 + K]
    ybig = torch.full((M, N + 13), 7.0, dtype=torch.bfloat16, device=DEV)
    yv = ybig[:, :N]
    sk.sgemm_bf16_skinny_ex(xv, W.to(DEV), yv)
    torch.cuda.synchronize()
    _check(x, W, yv.contiguous())
    assert torch.all(ybig[:, N:] == 7.0), "wrote outside y"


def test_guard_bands_untouched():
    M, N, K = 4, 1001, 2048
    x, W = _inputs(M, N, K, seed=15)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), -3.0, dtype=torch.bfloat16, device=DEV)
    y = buf[pad:pad + M * N].view(M, N)
    for split in (1, 3):
        plan = sk.sgemm_plan_select(N, K, M).copy(split_k=split)
        sk.sgemm_bf16_skinny_ex(x.to(DEV), W.to(DEV), y, plan=plan)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == -3.0) and torch.all(buf[pad + M * N:] == -3.0)
        _check(x, W, y)


def test_errors_reported_on_gpu():
    x = torch.zeros((1, 72), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((16, 72), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sk.SgemmError) as e:
        sk.sgemm_bf16_skinny_ex(x[:, 1:65], W[:, :64].contiguous())
    assert e.value.status == sk.SGEMM_ERR_MISALIGNED
    with pytest.raises(sk.SgemmError) as e:
        sk.sgemm_bf16_skinny(torch.zeros((1, 12), dtype=torch.bfloat16, device=DEV),
                             torch.zeros((4, 12), dtype=torch.bfloat16, device=DEV))
    assert e.value.status == sk.SGEMM_ERR_UNSUPPORTED_SHAPE
    # the context is still usable
    y = sk.sgemm_bf16_skinny(x[:, :64], W[:, :64].contiguous())
    torch.cuda.synchronize()
    assert torch.all(y == 0)


# ------------------------------------------------------- full-size, sampled rows
def _sample_rows(N, n=96, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(N, size=min(n, N), replace=False).tolist())
    rows |= {0, 1, N - 2, N - 1}
    return np.array(sorted(r for r in rows if 0 <= r < N))


@pytest.mark.parametrize("N,K", SWEEP_SHAPES + [(77440, 4096)])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_full_size_shapes_sampled(M, N, K):
    xd = synth.normal_bf16((M, K), synth.X_STD, seed=100 + M, device=DEV)
    Wd = synth.normal_bf16((N, K), synth.W_STD, seed=200, device=DEV)
    y = sk.sgemm_bf16_skinny(xd, Wd)
    torch.cuda.synchronize()
    rows = _sample_rows(N, seed=N)
    x = xd.cpu()
    Ws = Wd[torch.as_tensor(rows, device=DEV)].cpu()
    ref = oracle.skinny_gemm(synth.bits(x), synth.bits(Ws))
    rep = compare(synth.bits(y)[:, rows], ref, synth.bits(x), synth.bits(Ws))
    assert rep["ok"], rep


# --------------------------------------------------------------- batched pairs
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_batched_pairs_match_separate_calls(M):
    N, K = 4096, 128
    items, refs = [], []
    for i in range(2):
        x, W = _inputs(M, N, K, seed=300 + 10 * i, wstd=synth.PAIR_W_STD)
        items.append((x.to(DEV), W.to(DEV)))
        refs.append((x, W))
    plan = sk.sgemm_plan_select(N, K, M)
    outs = sk.sgemm_bf16_skinny_batched(items)
    torch.cuda.synchronize()
    for (xd, Wd), y, (x, W) in zip(items, outs, refs):
        sep = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
        torch.cuda.synchronize()
        assert torch.equal(sep.view(torch.int16), y.view(torch.int16)), "pair != separate call"
        _check(x, W, y)


def test_batched_strided_view_inputs():
    """x_i as a narrow -> unflatten -> transpose view of one activation buffer
    (the view pattern of the paired-projection page), batch of 2 and of 8."""
    M, N, K = 3, 4096, 128
    for batch in (2, 8):
        act = synth.normal_bf16((M, batch * K), 1.0, seed=400 + batch).to(DEV)
        xs = act.unflatten(1, (batch, K)).transpose(0, 1)  # [batch, M, K], row stride batch*K
        Ws = [synth.normal_bf16((N, K), synth.PAIR_W_STD, seed=500 + i).to(DEV)
              for i in range(batch)]
        outs = sk.sgemm_bf16_skinny_batched([(xs[i], Ws[i]) for i in range(batch)])
        torch.cuda.synchronize()
        for i in range(batch):
            _check(xs[i].contiguous().cpu(), Ws[i].cpu(), outs[i])


def test_batched_with_split_k():
    M, N, K = 2, 1000, 4096
    items, refs = [], []
    for i in range(3):
        x, W = _inputs(M, N, K, seed=600 + i)
        items.append((x.to(DEV), W.to(DEV)))
        refs.append((x, W))
    plan = sk.sgemm_plan_select(N, K, M).copy(split_k=4)
    outs = sk.sgemm_bf16_skinny_batched_ex(items, plan=plan)
    torch.cuda.synchronize()
    for (xd, Wd), y, (x, W) in zip(items, outs, refs):
        sep = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
        torch.cuda.synchronize()
        assert torch.equal(sep.view(torch.int16), y.view(torch.int16))
        _check(x, W, y)


# ---------------------------------------------------------------- CUDA graphs
@pytest.mark.parametrize("split", [1, 2])
def test_graph_replay_and_in_place_weight_refresh(split):
    """Capture, replay, then refresh W in place and replay again: the graph
    must see the new weights (the library keeps no copy of W)."""
    M, N, K = 2, 2048, 4096
    x, W = _inputs(M, N, K, seed=700)
    xd, Wd = x.to(DEV), W.to(DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    plan = sk.sgemm_plan_select(N, K, M).copy(split_k=split)
    sk.sgemm_bf16_skinny_ex(xd, Wd, y, plan=plan)  # eager warm-up (allocates scratch)
    torch.cuda.synchronize()
    eager = y.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sk.sgemm_bf16_skinny_ex(xd, Wd, y, plan=plan)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), eager.view(torch.int16))
    W2 = synth.normal_bf16((N, K), synth.W_STD, seed=701)
    Wd.copy_(W2.to(DEV))
    g.replay()
    torch.cuda.synchronize()
    _check(x, W2, y)


def test_batched_graph_replay():
    M, N, K = 1, 4096, 128
    items = []
    for i in range(2):
        x, W = _inputs(M, N, K, seed=800 + i, wstd=synth.PAIR_W_STD)
        items.append((x.to(DEV), W.to(DEV), torch.empty((M, N), dtype=torch.bfloat16, device=DEV)))
    sk.sgemm_bf16_skinny_batched(items)
    torch.cuda.synchronize()
    eager = [it[2].clone() for it in items]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sk.sgemm_bf16_skinny_batched(items)
    for it in items:
        it[2].zero_()
    g.replay()
    torch.cuda.synchronize()
    for it, e in zip(items, eager):
        assert torch.equal(it[2].view(torch.int16), e.view(torch.int16))


# ------------------------------------------- plan equivalence and launch flags
@pytest.mark.parametrize("M", [1, 3, 4])
def test_plans_with_same_lanes_per_row_agree_bitwise(M):
    """For the CUDA-core kernels the accumulation order depends only on (K range,
    lanes per row, FMA pairing): the mixed-precision FMA and the widened FP32
    FMA, any R, U and CTA size must give the same bits (and so must any packed
    FP32x2 plans among themselves, and any diagonal-MMA plans among
    themselves).  For the mma.sync kernels it depends on (K range, warps per
    CTA), for the tcgen05 kernel on (K range, split): any U, batch depth and
    ring must give the same bits."""
    N, K = 1500, 3072
    x, W = _inputs(M, N, K, seed=31)
    xd, Wd = x.to(DEV), W.to(DEV)
    by_lpr = {}
    for p in _all_plans():
        for split in (1, 2):
            plan = p.copy(split_k=split)
            if sk.sgemm_plan_check(plan, M, N, K) != sk.SGEMM_OK:
                continue
            y = sk.sgemm_bf16_skinny_ex(xd, Wd, plan=plan)
            torch.cuda.synchronize()
            mma = plan.variant in (sk.SGEMM_VARIANT_MMA, sk.SGEMM_VARIANT_TC05)
            # the widened and the mixed-precision FMA round identically; the packed
            # FP32x2 FMA keeps two partial sums, a different order of its own
            ffma2 = plan.variant in (sk.SGEMM_VARIANT_LDG_FFMA2, sk.SGEMM_VARIANT_LDGX_FFMA2)
            diag = plan.variant == sk.SGEMM_VARIANT_LDG_MMA  # its own fixed order
            fam = plan.variant if (mma or diag) else (5 if ffma2 else -1)
            key = (fam, plan.lanes_per_row, split, plan.threads if mma else 0)
            if key in by_lpr:
                assert torch.equal(by_lpr[key][1].view(torch.int16), y.view(torch.int16)), \
                    (by_lpr[key][0], plan)
            else:
                by_lpr[key] = (plan, y)
    for _, (plan, y) in by_lpr.items():
        _check(x, W, y)


def _chain(xd, Ws, flags, plan_split=1):
    """y_i = x_i W_i^T where x_{i+1} is a rescaled copy of y_i (a dependent chain)."""
    outs = []
    x = xd
    for W in Ws:
        N, K = W.shape
        plan = sk.sgemm_plan_select(N, K, x.shape[0]).copy(split_k=plan_split)
        y = torch.empty((x.shape[0], N), dtype=torch.bfloat16, device=DEV)
        sk.sgemm_bf16_skinny_ex(x, W, y, plan=plan, flags=flags)
        outs.append(y)
        x = (y[:, :K].float() * 8.0).to(torch.bfloat16)  # next input depends on this output
    return outs


@pytest.mark.parametrize("flags", [sk.SGEMM_FLAG_PDL,
                                   sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY])
@pytest.mark.parametrize("split", [1, 3])
def test_pdl_chain_matches_plain_launches(flags, split):
    M = 2
    shapes = [(4096, 4096), (4096, 4096), (2048, 4096), (4096, 2048)]
    Ws = [synth.normal_bf16(s, synth.W_STD, seed=40 + i).to(DEV) for i, s in enumerate(shapes)]
    xd = synth.normal_bf16((M, 4096), 1.0, seed=39).to(DEV)
    ref = _chain(xd, Ws, 0, split)
    torch.cuda.synchronize()
    got = _chain(xd, Ws, flags, split)
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # and under graph capture
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gout = _chain(xd, Ws, flags, split)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, gout):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
