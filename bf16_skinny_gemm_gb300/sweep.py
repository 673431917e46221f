"""Offline plan sweep: time every compiled plan on each decode shape and write
the fastest into ``csrc/plan_table.inc``.

Protocol (after vLLM PR #62949, Details: "a CUDA-graph sweep over block_size,
outputs_per_block, k_unroll, vector_width ... with the weight rotated out of
L2", and PR #65306, Validation: a chain over copies of the weight adding up to
at least 1 GiB, captured in a CUDA graph, trials interleaved):

- for each (N, K): R weight copies with R * |W| >= max(1 GiB, 4 x L2), so every
  GEMM of a chain reads its weights from HBM;
- for each M and each candidate plan (every compiled kernel configuration x
  CTA size x split factor): one CUDA graph of R GEMMs through the public
  ``sgemm_bf16_skinny_ex`` call, launched with the decode-chain launch flags
  (programmatic dependent launch, weights read-only);
- T trials of P replays each, interleaved across candidates; before every
  timed replay a separate buffer of several GiB is read, so each replay starts
  from the state a decode step leaves behind (caches and address translations
  filled by other data; a clean read, so nothing is written back during the
  timed replay).  Replaying one graph back to back instead lets part of the
  weight set and its translations survive from the previous replay, which
  flatters the CUDA-core streaming kernels by about 10 %.  The score is the
  median per-GEMM time.  The fastest candidate is kept.  (The pages keep a
  plan only if it beats cuBLAS by 5 %; here there is no other library to fall
  back to, so the table keeps the fastest plan outright.)

The batched pair shape (4096, 128) is swept as it is used: two problems per
launch.

Usage (on the GPU):
    python -m bf16_skinny_gemm_gb300.sweep --out bf16_skinny_gemm_gb300/csrc/plan_table.inc
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import time

import torch

import bf16_skinny_gemm_gb300 as sk
from bf16_skinny_gemm_gb300 import synth

DECODE_SHAPES = [(12576, 4096), (4096, 4096), (2048, 4096), (4096, 1024), (8192, 1536),
                 (4096, 8192), (77440, 4096), (288, 4096)]
PAIR_SHAPE = (4096, 128)
HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_OUT = os.path.join(HERE, "csrc", "plan_table.inc")


# TMA + tcgen05 kernel: (ring slots, 64-element boxes per stage), cluster splits of K,
# and CTAs per SM of the persistent grid (split 1 only)
TC05_GEOMETRY = [(4, 1), (6, 1), (8, 1), (12, 1), (2, 2), (3, 2), (4, 2), (6, 2), (2, 3), (3, 3), (4, 3), (2, 4), (3, 4)]
TC05_SPLITS = [1, 2, 3, 4, 6, 8, 16]
TC05_CTAS = [0, 1, 2]
# cluster-split streaming plans: CTAs of a cluster sharing a row range's K
LDG_CLUSTER_SPLITS = [2, 3, 4, 6, 8]


def candidates(M, N, K, splits, ctas=(0,)):
    """Every compiled plan x split (and x CTAs per SM of the grid, `ctas`; 0 =
    the occupancy limit) that can run (M, N, K)."""
    out = []
    for i in range(sk.sgemm_plan_count()):
        base = sk.sgemm_plan_get(i)
        if base.variant == sk.SGEMM_VARIANT_LDG_CLUSTER:
            variants = [base.copy(split_k=s) for s in LDG_CLUSTER_SPLITS]
        elif base.variant == sk.SGEMM_VARIANT_TC05:
            if base.k_unroll != 1:
                continue  # the enumeration lists this kernel twice; its geometry is swept here
            variants = [base.copy(stages=r, k_unroll=nb, split_k=s, ctas_per_sm=c)
                        for r, nb in TC05_GEOMETRY for s in TC05_SPLITS
                        for c in (TC05_CTAS if s == 1 else [0])]
        else:
            variants = [base.copy(split_k=s, ctas_per_sm=c) for s in splits for c in ctas]
        for p in variants:
            if sk.sgemm_plan_check(p, M, N, K) == sk.SGEMM_OK:
                out.append(p)
    return out


def sweep_shape(N, K, Ms, splits, flags, trials, replays, min_bytes, pair=False, log=print,
                prefilter=0, prefilter_bytes=0.0, ctas=(0,), cold=None):
    """Time every candidate plan of (N, K) for each M; returns {M: result}.

    prefilter = P > 0 times the candidates in two stages: first all of them
    (weight copies totalling ``prefilter_bytes``) with 2 trials x 3 replays,
    then the P fastest (and the heuristic plan) with the full protocol; the
    winner comes from the second stage.
    """
    dev = torch.device("cuda")
    R = max(2, math.ceil(min_bytes / (2 * N * K)))
    if pair:
        R += R % 2
    std = synth.PAIR_W_STD if pair else synth.W_STD
    W = torch.empty((R, N, K), dtype=torch.bfloat16, device=dev)
    for i in range(R):
        W[i].copy_(synth.normal_bf16((N, K), std, seed=i, device=dev))
    results = {}

    def same(a, b):
        da, db = a.as_dict(), b.as_dict()
        da.pop("id"), db.pop("id")
        return da == db

    for M in Ms:
        x = synth.normal_bf16((R, M, K), synth.X_STD, seed=1000 + M, device=dev)
        y = torch.empty((R, M, N), dtype=torch.bfloat16, device=dev)
        cands = candidates(M, N, K, splits, ctas)
        heur = sk.sgemm_plan_select(N, K, M)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())

        def chain(plan, fl, n):
            if pair:
                for i in range(0, n, 2):
                    sk.sgemm_bf16_skinny_batched_ex([(x[i], W[i], y[i]), (x[i + 1], W[i + 1], y[i + 1])],
                                                    plan=plan, flags=fl)
            else:
                for i in range(n):
                    sk.sgemm_bf16_skinny_ex(x[i], W[i], y[i], plan=plan, flags=fl)

        def time_plans(plans, n, n_trials, n_replays):
            """Median µs per launch of each plan over a graph of n GEMMs."""
            for p in plans:
                chain(p, 0, n)  # eager once (split-K scratch is allocated outside capture)
            torch.cuda.synchronize()
            graphs = []
            for p in plans:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        chain(p, flags, n)
                graphs.append(g)
            torch.cuda.current_stream().wait_stream(s)
            for g in graphs:
                g.replay()
                g.replay()
            torch.cuda.synchronize()
            times = [[] for _ in plans]
            per_launch = n // 2 if pair else n
            for _ in range(n_trials):
                for ci, g in enumerate(graphs):
                    if cold is None:  # back-to-back replays
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record()
                        for _ in range(n_replays):
                            g.replay()
                        e1.record()
                        e1.synchronize()
                        times[ci].append(e0.elapsed_time(e1) * 1e3 / n_replays / per_launch)
                        continue
                    evs = []
                    for _ in range(n_replays):
                        cold.sum()  # not timed: caches and translations now hold other data
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record()
                        g.replay()
                        e1.record()
                        evs.append((e0, e1))
                    torch.cuda.synchronize()
                    times[ci] += [a.elapsed_time(b) * 1e3 / per_launch for a, b in evs]
            del graphs
            torch.cuda.synchronize()
            return [statistics.median(t) for t in times]

        stage1 = None
        if prefilter > 0 and len(cands) > prefilter:
            R1 = min(R, max(2, math.ceil(prefilter_bytes / (2 * N * K))))
            R1 += R1 % 2 if pair else 0
            med1 = time_plans(cands, R1, 2, 3)
            keep = sorted(range(len(cands)), key=lambda i: med1[i])[:prefilter]
            keep += [i for i, p in enumerate(cands) if same(p, heur) and i not in keep]
            stage1 = [(cands[i].as_dict(), round(med1[i], 3)) for i in
                      sorted(range(len(cands)), key=lambda i: med1[i])]
            cands = [cands[i] for i in keep]
        med = time_plans(cands, R, trials, replays)
        order = sorted(range(len(cands)), key=lambda i: med[i])
        best = cands[order[0]]
        nbytes = (2 if pair else 1) * 2 * (N * K + M * K + M * N)
        heur_us = next((med[i] for i, p in enumerate(cands) if same(p, heur)), None)
        results[M] = {"plan": best.as_dict(), "us": med[order[0]],
                      "gbs": nbytes / med[order[0]] / 1e3,
                      "heuristic_us": heur_us,
                      "top": [(cands[i].as_dict(), round(med[i], 3)) for i in order[:5]],
                      "all": [(cands[i].as_dict(), round(med[i], 3)) for i in order],
                      "copies": R, "candidates": len(cands)}
        if stage1 is not None:
            results[M]["prefilter"] = stage1
        log(f"  N={N} K={K} M={M}: best {med[order[0]]:.3f} us "
            f"({results[M]['gbs']:.0f} GB/s) {_short(best)}; heuristic "
            f"{heur_us if heur_us is None else round(heur_us, 3)} us; {len(cands)} candidates"
            + ("" if stage1 is None else f" (of {len(stage1)} prefiltered)"))
    del W
    torch.cuda.empty_cache()
    return results


def _short(p):
    return (f"v{p.variant} t{p.threads} R{p.rows_per_warp} L{p.lanes_per_row} "
            f"U{p.k_unroll}x{max(p.stages, 1)} S{p.split_k}")


def read_table(path):
    """Entries of an existing generated table: {(N, K, M): {"plan": ..., "us", "gbs"}}."""
    out = {}
    keys = ["variant", "threads", "rows_per_warp", "lanes_per_row", "k_unroll", "split_k",
            "stages", "ctas_per_sm"]
    with open(path) as f:
        for ln in f:
            ln = ln.strip()
            if not ln.startswith("{"):
                continue
            body, _, comment = ln.partition("//")
            vals = [int(v) for v in body.strip().strip("{},").split(",")]
            N, K, M = vals[:3]
            plan = dict(zip(keys, vals[3:]))
            plan.update(vec_bytes=16, id=-1)
            us = float(comment.split("us")[0]) if "us" in comment else 0.0
            gbs = float(comment.split(",")[1].split("GB/s")[0]) if "GB/s" in comment else 0.0
            out[(N, K, M)] = {"plan": plan, "us": us, "gbs": gbs}
    return out


def write_table(entries, path, note):
    lines = [
        "// Generated by bf16_skinny_gemm_gb300/sweep.py -- do not edit by hand.",
        f"// {note}",
        "// Fields: N, K, M, variant, threads, R, LPR, U, split, stages, ctas_per_sm",
    ]
    for (N, K, M), r in sorted(entries.items()):
        p = r["plan"]
        lines.append(
            f"{{{N}, {K}, {M}, {p['variant']}, {p['threads']}, {p['rows_per_warp']}, "
            f"{p['lanes_per_row']}, {p['k_unroll']}, {p['split_k']}, {p['stages']}, "
            f"{p['ctas_per_sm']}}},  // {r['us']:.3f} us, {r['gbs']:.0f} GB/s")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--out", default=DEFAULT_OUT)
    ap.add_argument("--json", default=None, help="also write all timings here")
    ap.add_argument("--ms", default="1,2,3,4")
    ap.add_argument("--splits", default="1,2,4")
    ap.add_argument("--cold-gib", type=float, default=4.0,
                    help="GiB of other memory read before each timed replay (0 = replay "
                         "back to back)")
    ap.add_argument("--ctas", default="0",
                    help="CTAs per SM of the grid for the streaming and mma.sync plans "
                         "(0 = occupancy limit), e.g. 0,1,2")
    ap.add_argument("--trials", type=int, default=5)
    ap.add_argument("--replays", type=int, default=10)
    ap.add_argument("--min-bytes", type=float, default=float(1 << 30))
    ap.add_argument("--shapes", default=None, help="e.g. 4096x4096,2048x4096 (default: all)")
    ap.add_argument("--no-pair", action="store_true")
    ap.add_argument("--note", default="",
                    help="appended to the table's header line (where its entries came from)")
    ap.add_argument("--merge", default=None,
                    help="start from this existing table and replace only the swept entries")
    ap.add_argument("--prefilter", type=int, default=0,
                    help="time all candidates on a shorter cold chain first and keep this many "
                         "for the full protocol (0 = time every candidate fully)")
    args = ap.parse_args(argv)

    assert torch.cuda.is_available(), "the sweep runs on the GPU"
    sk.load()
    sk.sgemm_init()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    min_bytes = max(args.min_bytes, 4 * l2)
    Ms = [int(v) for v in args.ms.split(",")]
    splits = [int(v) for v in args.splits.split(",")]
    ctas = tuple(int(v) for v in args.ctas.split(","))
    cold = None
    if args.cold_gib > 0:
        cold = torch.ones(int(args.cold_gib * 2**30) // 8, dtype=torch.int64, device="cuda")
    flags = sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY
    shapes = DECODE_SHAPES
    if args.shapes:
        shapes = [tuple(int(v) for v in t.split("x")) for t in args.shapes.split(",")]
    t0 = time.time()
    entries, dump = ({}, {})
    if args.merge:
        entries = read_table(args.merge)
    for (N, K) in shapes:
        res = sweep_shape(N, K, Ms, splits, flags, args.trials, args.replays, min_bytes,
                          prefilter=args.prefilter, prefilter_bytes=min_bytes, ctas=ctas,
                          cold=cold)
        for M, r in res.items():
            entries[(N, K, M)] = r
            dump[f"{N}x{K}x{M}"] = r
    if not args.no_pair:
        N, K = PAIR_SHAPE
        res = sweep_shape(N, K, Ms, splits, flags, args.trials, args.replays, min_bytes, pair=True,
                          prefilter=args.prefilter, prefilter_bytes=min_bytes, ctas=ctas,
                          cold=cold)
        for M, r in res.items():
            entries[(N, K, M)] = r
            dump[f"{N}x{K}x{M}-pair"] = r
    note = (f"{torch.cuda.get_device_name(0)}, {len(entries)} entries, cold L2 (>= "
            f"{min_bytes / 2**30:.2f} GiB of weight copies per shape"
            + (f", {args.cold_gib:g} GiB of other memory read before each timed replay"
               if cold is not None else ", replays back to back")
            + f"), launch flags PDL|readonly, "
            f"{args.trials} interleaved trials x {args.replays} graph replays, median"
            + (f", top {args.prefilter} of a first pass (2 trials x 3 replays) timed fully"
               if args.prefilter else "")
            + (f"; {args.note}" if args.note else ""))
    write_table(entries, args.out, note)
    if args.json:
        with open(args.json, "w") as f:
            json.dump(dump, f, indent=1)
    print(f"wrote {args.out} ({len(entries)} entries) in {time.time() - t0:.0f} s")
    return 0


if __name__ == "__main__":
    sys.exit(main())
