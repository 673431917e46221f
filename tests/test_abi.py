"""The C-ABI library on a CPU-only machine: it loads, exports every function
the public header declares, and its host-side logic (argument checks, plan
selection and plan checks) behaves as documented.  No kernel is launched:
every call below returns before the library touches a CUDA device.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import bf16_skinny_gemm_gb300 as sk
from bf16_skinny_gemm_gb300 import build as skbuild

HEADER = os.path.join(skbuild.INCLUDE, "sgemm_skinny.h")


@pytest.fixture(scope="module")
def lib():
    skbuild.build()
    return sk.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(sgemm_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("sgemm_bf16_skinny", "sgemm_bf16_skinny_batched", "sgemm_plan_select"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings(lib):
    for s in range(7):
        assert sk.sgemm_status_string(s)
    assert sk.sgemm_status_string(99) == "unknown status"
    assert re.match(r"^\d+\.\d+\.\d+$", sk.sgemm_version())


# pointers that are never dereferenced: every call below fails validation first
A16 = 0x10000
NULL = None


def _call(lib, x, W, y, M, N, K, ldx=None, ldy=None):
    return lib.sgemm_bf16_skinny_ex(x, K if ldx is None else ldx, W, y, N if ldy is None else ldy,
                                    M, N, K, None, 0, None)


@pytest.mark.parametrize("M,N,K,expect", [
    (0, 16, 64, sk.SGEMM_ERR_INVALID_ARG),
    (9, 16, 64, sk.SGEMM_ERR_INVALID_ARG),
    (1, 0, 64, sk.SGEMM_ERR_INVALID_ARG),
    (1, 16, 0, sk.SGEMM_ERR_INVALID_ARG),
    (1, 16, 12, sk.SGEMM_ERR_UNSUPPORTED_SHAPE),
    (4, 16, 1001, sk.SGEMM_ERR_UNSUPPORTED_SHAPE),
])
def test_bad_shapes_rejected(lib, M, N, K, expect):
    assert _call(lib, A16, A16, A16, M, N, K) == expect


def test_null_pointers_rejected(lib):
    assert _call(lib, NULL, A16, A16, 1, 16, 64) == sk.SGEMM_ERR_INVALID_ARG
    assert _call(lib, A16, NULL, A16, 1, 16, 64) == sk.SGEMM_ERR_INVALID_ARG
    assert _call(lib, A16, A16, NULL, 1, 16, 64) == sk.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_bf16_skinny(A16, A16, NULL, 1, 16, 64, None) == sk.SGEMM_ERR_INVALID_ARG


def test_bad_strides_and_alignment_rejected(lib):
    assert _call(lib, A16, A16, A16, 2, 16, 64, ldx=56) == sk.SGEMM_ERR_INVALID_ARG
    assert _call(lib, A16, A16, A16, 2, 16, 64, ldy=15) == sk.SGEMM_ERR_INVALID_ARG
    assert _call(lib, A16, A16, A16, 2, 16, 64, ldx=68) == sk.SGEMM_ERR_MISALIGNED
    assert _call(lib, A16 + 8, A16, A16, 1, 16, 64) == sk.SGEMM_ERR_MISALIGNED
    assert _call(lib, A16, A16 + 2, A16, 1, 16, 64) == sk.SGEMM_ERR_MISALIGNED
    assert _call(lib, A16, A16, A16 + 1, 1, 16, 64) == sk.SGEMM_ERR_MISALIGNED


def test_fused_chain_epilogue_argument_checks(lib):
    X, W, Y, XN = 0x10000, 0x20000, 0x30000, 0x40000

    def call(xn, ldn, n_next, y=Y, x=X):
        return lib.sgemm_bf16_skinny_rescale_ex(x, 64, W, y, 16, 2, 16, 64, xn, ldn, n_next, 0.5,
                                                None, 0, None)
    assert call(NULL, 64, 64) == sk.SGEMM_ERR_INVALID_ARG
    assert call(XN, 64, 0) == sk.SGEMM_ERR_INVALID_ARG            # n_next < 1
    assert call(XN, 32, 64) == sk.SGEMM_ERR_INVALID_ARG           # row stride < n_next
    assert call(XN, 64, 1 << 31) == sk.SGEMM_ERR_INVALID_ARG      # n_next must fit an int
    assert call(XN + 1, 64, 64) == sk.SGEMM_ERR_MISALIGNED
    # x_next may overlap none of x, W and y: the kernel still reads x and W
    assert call(X + 64, 64, 64) == sk.SGEMM_ERR_INVALID_ARG       # inside x
    assert call(W + 2 * 16 * 64 - 2, 64, 64) == sk.SGEMM_ERR_INVALID_ARG  # last W element
    assert call(Y, 64, 64) == sk.SGEMM_ERR_INVALID_ARG
    assert call(X - 2 * (64 + 64) + 2, 64, 64) == sk.SGEMM_ERR_INVALID_ARG  # ends inside x
    # the problem's own checks still come first
    assert lib.sgemm_bf16_skinny_rescale_ex(X, 64, W, Y, 16, 9, 16, 64, XN, 64, 64, 0.5, None, 0,
                                            None) == sk.SGEMM_ERR_INVALID_ARG


def test_fp32_output_argument_checks(lib):
    X, W, Y = 0x10000, 0x20000, 0x30000
    f = lib.sgemm_bf16_skinny_f32out_ex
    assert f(X, 64, W, Y + 2, 16, 1, 16, 64, None, 0, None) == sk.SGEMM_ERR_MISALIGNED
    assert f(X, 64, W, NULL, 16, 1, 16, 64, None, 0, None) == sk.SGEMM_ERR_INVALID_ARG
    assert f(X, 64, W, Y, 15, 2, 16, 64, None, 0, None) == sk.SGEMM_ERR_INVALID_ARG
    assert f(X, 64, W, Y, 16, 1, 16, 60, None, 0, None) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE


def test_unknown_flags_rejected(lib):
    assert lib.sgemm_bf16_skinny_ex(A16, 64, A16, A16, 16, 1, 16, 64, None, 8, None) == \
        sk.SGEMM_ERR_INVALID_ARG
    pairs = (sk.Pair * 1)()
    pairs[0].x, pairs[0].W, pairs[0].y, pairs[0].ldx, pairs[0].ldy = A16, A16, A16, 64, 16
    assert lib.sgemm_bf16_skinny_batched_ex(pairs, 1, 1, 16, 64, None, 8, None) == \
        sk.SGEMM_ERR_INVALID_ARG


def test_batched_argument_checks(lib):
    pairs = (sk.Pair * 9)()
    for p in pairs:
        p.x, p.W, p.y, p.ldx, p.ldy = A16, A16, A16, 64, 16
    assert lib.sgemm_bf16_skinny_batched(pairs, 0, 1, 16, 64, None) == sk.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_bf16_skinny_batched(pairs, 9, 1, 16, 64, None) == sk.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_bf16_skinny_batched(None, 2, 1, 16, 64, None) == sk.SGEMM_ERR_INVALID_ARG
    pairs[1].W = A16 + 4
    assert lib.sgemm_bf16_skinny_batched(pairs, 2, 1, 16, 64, None) == sk.SGEMM_ERR_MISALIGNED


def test_bad_plans_rejected(lib):
    # a streaming-kernel plan (the tcgen05 plans have their own test below)
    good = next(p for p in (sk.sgemm_plan_get(i) for i in range(sk.sgemm_plan_count()))
                if p.variant == sk.SGEMM_VARIANT_LDG_MIXFMA and p.k_unroll == 8)
    assert sk.sgemm_plan_check(good, 1, 4096, 4096) == sk.SGEMM_OK
    for change in ({"variant": 7}, {"variant": -1}, {"variant": 3}, {"variant": 4}, {"variant": 8},
                   {"threads": 48}, {"threads": 512}, {"vec_bytes": 8},
                   {"split_k": 0}, {"k_unroll": 3}, {"lanes_per_row": 4}, {"stages": 3}):
        bad = good.copy(**change)
        assert sk.sgemm_plan_check(bad, 1, 4096, 4096) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE, change
        assert _call_plan(lib, bad) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE, change
    # more splits than chunks of K
    assert sk.sgemm_plan_check(good.copy(split_k=9), 1, 16, 64) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE


def _call_plan(lib, plan):
    return lib.sgemm_bf16_skinny_ex(A16, 4096, A16, A16, 4096, 1, 4096, 4096,
                                    ctypes.byref(plan), 0, None)


def test_plan_enumeration(lib):
    n = sk.sgemm_plan_count()
    assert n >= 8
    seen = set()
    for i in range(n):
        p = sk.sgemm_plan_get(i)
        key = tuple(p.as_dict().items())
        assert key not in seen
        seen.add(key)
        for M in range(1, 9):
            assert sk.sgemm_plan_check(p, M, 4096, 4096) == sk.SGEMM_OK, p
    with pytest.raises(sk.SgemmError):
        sk.sgemm_plan_get(n)


SHAPES = [(12576, 4096), (4096, 4096), (2048, 4096), (4096, 1024), (8192, 1536), (4096, 8192),
          (77440, 4096), (4096, 128), (1, 8), (300, 100000)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
def test_selected_plans_are_runnable(lib, N, K, M):
    p = sk.sgemm_plan_select(N, K, M)
    assert sk.sgemm_plan_check(p, M, N, K) == sk.SGEMM_OK, p
    # deterministic selection
    assert p.as_dict() == sk.sgemm_plan_select(N, K, M).as_dict()


def test_plan_select_out_of_range_still_returns_a_plan(lib):
    p = sk.sgemm_plan_select(-1, -1, 9)
    assert p.threads > 0 and p.id == -1


def test_heuristic_plan_splits_k_when_rows_leave_sms_idle(lib):
    # (320, 4096) at M = 1..4 has no table entry: 40 CTAs of rows alone would
    # leave most of 152 SMs idle, so K is split (down to 512 elements a split)
    for M in (1, 2, 3, 4):
        p = sk.sgemm_plan_select(320, 4096, M)
        assert p.id == -1 and p.split_k >= 4, p
        assert sk.sgemm_plan_check(p, M, 320, 4096) == sk.SGEMM_OK
    # enough rows: no extra split
    assert sk.sgemm_plan_select(100000, 4096, 1).split_k == 1
    # M >= 5 without a table entry: the 16-row tensor-core kernel
    for M in (5, 8):
        p = sk.sgemm_plan_select(3000, 2000, M)
        assert p.id == -1 and p.variant == sk.SGEMM_VARIANT_MMA, p
        assert sk.sgemm_plan_check(p, M, 3000, 2000) == sk.SGEMM_OK


def _tc05_plan():
    for i in range(sk.sgemm_plan_count()):
        p = sk.sgemm_plan_get(i)
        if p.variant == sk.SGEMM_VARIANT_TC05:
            return p
    raise AssertionError("no TC05 plan enumerated")


def test_tc05_plan_checks(lib):
    """Host-side checks of the TMA + tcgen05 plans: fixed geometry (192
    threads, 128-row tiles), 1..4 boxes per stage, 2..16 ring slots that fit
    shared memory, and a cluster split of 1..16 with at least one 64-element
    box of K per split."""
    p = _tc05_plan()
    assert (p.threads, p.rows_per_warp, p.lanes_per_row) == (192, 128, 0)
    for M in range(1, 9):
        assert sk.sgemm_plan_check(p, M, 4096, 4096) == sk.SGEMM_OK
    for split in (1, 2, 3, 5, 8, 16):
        assert sk.sgemm_plan_check(p.copy(split_k=split), 4, 613, 2600) == sk.SGEMM_OK
    for change in ({"threads": 256}, {"rows_per_warp": 64}, {"lanes_per_row": 32},
                   {"k_unroll": 0}, {"k_unroll": 5}, {"k_unroll": 8}, {"stages": 1}, {"stages": 17},
                   {"split_k": 0}, {"split_k": 17}, {"ctas_per_sm": -1}, {"vec_bytes": 8},
                   {"stages": 16, "k_unroll": 4}):
        bad = p.copy(**change)
        assert sk.sgemm_plan_check(bad, 1, 4096, 4096) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE, change
        assert _call_plan(lib, bad) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE, change
    # K = 64 is one box: no split; K = 72 is two boxes
    assert sk.sgemm_plan_check(p.copy(split_k=2), 1, 16, 64) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE
    assert sk.sgemm_plan_check(p.copy(split_k=2), 1, 16, 72) == sk.SGEMM_OK
    # the largest ring that fits: 12 single-box stages (12 x 18 KiB + slack)
    assert sk.sgemm_plan_check(p.copy(stages=12, k_unroll=1), 8, 4096, 4096) == sk.SGEMM_OK
    assert sk.sgemm_plan_check(p.copy(stages=6, k_unroll=2, split_k=16), 8, 4096, 4096) == \
        sk.SGEMM_ERR_UNSUPPORTED_SHAPE  # plus 15 x 8 x 128 floats of cluster partials


def test_plan_table_round_trip(tmp_path):
    """The sweep's table writer and reader (used by --merge) agree, and the
    compiled table parses: every entry is a plan the library accepts."""
    from bf16_skinny_gemm_gb300 import sweep
    entries = sweep.read_table(os.path.join(skbuild.CSRC, "plan_table.inc"))
    assert len(entries) >= 32
    for (N, K, M), r in entries.items():
        plan = sk.Plan(**{**r["plan"], "id": -1})
        assert sk.sgemm_plan_check(plan, M, N, K) == sk.SGEMM_OK, (N, K, M, r["plan"])
        assert sk.sgemm_plan_select(N, K, M).id >= 0, (N, K, M)
    out = tmp_path / "table.inc"
    sweep.write_table(entries, str(out), "round trip")
    again = sweep.read_table(str(out))
    assert again.keys() == entries.keys()
    for k in entries:
        assert again[k]["plan"] == entries[k]["plan"]
        assert abs(again[k]["us"] - entries[k]["us"]) < 1e-3


def test_noalloc_plan_substitutions(lib):
    """The plan the no-allocation split-K call runs: the selected plan with the
    requested split, except for plans that do not split K through scratch."""
    def kernel(variant, **kw):
        for i in range(sk.sgemm_plan_count()):
            p = sk.sgemm_plan_get(i)
            if p.variant == variant and all(getattr(p, k) == v for k, v in kw.items()):
                return p
        raise AssertionError((variant, kw))

    # an ordinary streaming plan keeps everything but split_k
    base = kernel(sk.SGEMM_VARIANT_LDG_MIXFMA)
    st, p = sk.sgemm_splitk_noalloc_plan(4096, 4096, 2, 3, base)
    assert st == sk.SGEMM_OK and p.as_dict() == base.copy(split_k=3).as_dict()
    # tcgen05 plans (their split reduces in a cluster) -> the CUDA-core streaming plan
    st, p = sk.sgemm_splitk_noalloc_plan(4096, 4096, 4, 4, kernel(sk.SGEMM_VARIANT_TC05))
    assert st == sk.SGEMM_OK
    assert (p.variant, p.threads, p.rows_per_warp, p.lanes_per_row, p.k_unroll, p.stages,
            p.split_k) == (sk.SGEMM_VARIANT_LDG_MIXFMA, 256, 1, 32, 8, 1, 4), p
    # a 16-row tensor-core plan keeps its kernel
    mma = kernel(sk.SGEMM_VARIANT_MMA)
    st, p = sk.sgemm_splitk_noalloc_plan(4096, 4096, 4, 2, mma)
    assert st == sk.SGEMM_OK and p.as_dict() == mma.copy(split_k=2).as_dict()
    # the selected plan by default; split_k below 2 is refused
    st, p = sk.sgemm_splitk_noalloc_plan(4096, 8192, 1, 4)
    assert st == sk.SGEMM_OK and p.split_k == 4
    assert sk.sgemm_splitk_noalloc_plan(4096, 8192, 1, 1)[0] == sk.SGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("N,K,M", [(4096, 8192, 1), (2048, 4096, 4), (77440, 4096, 8), (1, 8, 1)])
def test_sweep_candidates_are_valid_plans(lib, N, K, M):
    """Every plan the offline sweep would time passes the library's own plan
    check, no retired variant (3, 4, 8) appears, and the tcgen05 candidates
    cover 1..4 boxes per stage."""
    from bf16_skinny_gemm_gb300 import sweep

    cands = sweep.candidates(M, N, K, [1, 2, 4])
    assert cands
    for p in cands:
        assert sk.sgemm_plan_check(p, M, N, K) == sk.SGEMM_OK, p
        assert p.variant not in (3, 4, 8), p
    tc = [p for p in cands if p.variant == sk.SGEMM_VARIANT_TC05]
    assert {p.k_unroll for p in tc} == {1, 2, 3, 4}
    assert {p.stages for p in tc} >= {2, 3, 4}


def test_ldg_cluster_plan_checks(lib):
    """The cluster-split streaming plans (variant 11): the cluster instantiations
    of mixed-precision streaming configurations, at most 8 CTAs per cluster."""
    cl = next(p for p in (sk.sgemm_plan_get(i) for i in range(sk.sgemm_plan_count()))
              if p.variant == sk.SGEMM_VARIANT_LDG_CLUSTER)
    base = cl.copy(variant=sk.SGEMM_VARIANT_LDG_MIXFMA)
    for split in (1, 2, 3, 4, 8):
        assert sk.sgemm_plan_check(cl.copy(split_k=split), 4, 2048, 4096) == sk.SGEMM_OK, split
    assert sk.sgemm_plan_check(cl.copy(split_k=9), 4, 2048, 4096) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE
    # a configuration compiled only for other variants is refused
    mma = next(p for p in (sk.sgemm_plan_get(i) for i in range(sk.sgemm_plan_count()))
               if p.variant == sk.SGEMM_VARIANT_MMA)
    assert sk.sgemm_plan_check(mma.copy(variant=sk.SGEMM_VARIANT_LDG_CLUSTER, split_k=2), 4,
                               2048, 4096) == sk.SGEMM_ERR_UNSUPPORTED_SHAPE
    # the no-allocation call runs such a plan as variant 1 through its array
    st, p = sk.sgemm_splitk_noalloc_plan(2048, 4096, 2, 4, cl.copy(split_k=2))
    assert st == sk.SGEMM_OK and p.as_dict() == base.copy(split_k=4).as_dict()
