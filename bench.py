"""Cold-L2 benchmark of the GB300 BF16 skinny GEMM.

Default workload (one "step"): the decode-shape sweep at M = 1, 2, 4 over the
local (N, K) shapes (12576,4096), (4096,4096), (2048,4096), (4096,1024),
(8192,1536), (4096,8192).  Following the measurement protocol of vLLM PR
#65306 (Validation: each case is a chain over copies of the weight adding up to
at least 1 GiB, captured in a CUDA graph) and PR #62949 (Validation: cold-L2
numbers, the weight rotated out of L2), every (shape, M) is a CUDA graph of R
GEMMs, each on its own weight copy, with R copies totalling
>= max(1 GiB, 4 x L2).  So every GEMM reads its weights from HBM.

Reported (one JSON line on rank 0):
- value: algorithmic bytes (W + x + y) of the whole step / device time, GB/s,
  summed over ranks (replicas: each GPU runs the whole sweep);
- detail: per (N, K, M) cold-L2 us per GEMM, GB/s and fraction of HBM peak;
- roofline: the skinny kernel's achieved GB/s against the measured HBM peak;
- e2e: the same metric with every step's x copied in from pinned host memory
  and every y copied back, through the library's public call;
- cpu_baseline: the CPU oracle timed on a bounded sample on this host.

``--impl reference`` times the CPU oracle alone (the reference arm).
``--workload`` selects other configurations: single, lmhead, pairs, chain.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "cold-L2 GB/s and µs per GEMM at M=1/2/4; fraction of GB300 HBM peak"
SWEEP_SHAPES = [(12576, 4096), (4096, 4096), (2048, 4096), (4096, 1024), (8192, 1536),
                (4096, 8192)]
SWEEP_MS = [1, 2, 4]
LMHEAD = (77440, 4096)
PAIR = (4096, 128)
CHAIN = [((12576, 4096), 34), ((4096, 4096), 34), ((2048, 4096), 53), ((4096, 1024), 42),
         ((8192, 1536), 11), ((4096, 8192), 11), ((77440, 4096), 1)]
FALLBACK_HBM_GBS = 6800.0


def gemm_bytes(M, N, K):
    """Algorithmic bytes of one GEMM: W + x + y, BF16."""
    return 2 * (N * K + M * K + M * N)


# --------------------------------------------------------------------- helpers
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Dist:
    def __init__(self, torch, backend=None):
        self.torch = torch
        self.ws, self.rank, self.local = dist_info()
        self.pg = None
        if self.ws > 1:
            import torch.distributed as td
            backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
            td.init_process_group(backend=backend)
            self.td = td
            self.backend = backend

    def barrier(self):
        if self.ws > 1:
            self.td.barrier()

    def max(self, v: float) -> float:
        if self.ws == 1:
            return v
        t = self.torch.tensor([v], dtype=self.torch.float64,
                              device="cuda" if self.backend == "nccl" else "cpu")
        self.td.all_reduce(t, op=self.td.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v: float) -> float:
        if self.ws == 1:
            return v
        t = self.torch.tensor([v], dtype=self.torch.float64,
                              device="cuda" if self.backend == "nccl" else "cpu")
        self.td.all_reduce(t, op=self.td.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.ws > 1:
            self.td.destroy_process_group()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bf16_skinny_gemm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and not name.startswith("."):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch recorded from an ncu capture, keyed (N, K, M);
    ignored when the kernel sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic_skinny_gemm.txt")
    out, src = {}, None
    try:
        with open(path) as f:
            for ln in f:
                ln = ln.strip()
                if ln.startswith("kernel_source_sha256:"):
                    src = ln.split(":", 1)[1].strip()
                elif ln and not ln.startswith("#") and ln[0].isdigit():
                    p = ln.split()
                    out[(int(p[0]), int(p[1]), int(p[2]))] = float(p[3])
    except OSError:
        return {}, "no capture recorded"
    if src != kernel_source_hash():
        return {}, "kernel changed since the capture"
    return out, "ncu"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.splitlines():
            p = [v.strip() for v in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for name, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ workloads
class GraphSet:
    """Per (N, K, M): R GEMMs on R weight copies, captured in one CUDA graph.
    All x inputs of a step live in one packed buffer and all y outputs in
    another, so the end-to-end run moves them with one copy each way."""

    def __init__(self, torch, sk, synth, cases, min_bytes, seed=0, pairs=False):
        self.torch, self.sk = torch, sk
        dev = torch.device("cuda")
        self.cases = []
        self.weights = {}
        for (N, K) in sorted({(c[0], c[1]) for c in cases}, key=lambda s: -s[0] * s[1]):
            wbytes = 2 * N * K
            R = max(2, math.ceil(min_bytes / wbytes))
            std = synth.PAIR_W_STD if pairs else synth.W_STD
            ws = torch.empty((R, N, K), dtype=torch.bfloat16, device=dev)
            for i in range(R):
                ws[i].copy_(synth.normal_bf16((N, K), std, seed=seed + i, device=dev))
            self.weights[(N, K)] = ws
        x_elems = sum(self.weights[(N, K)].shape[0] * M * K for (N, K, M) in cases)
        y_elems = sum(self.weights[(N, K)].shape[0] * M * N for (N, K, M) in cases)
        self.x_pack = torch.empty(x_elems, dtype=torch.bfloat16, device=dev)
        self.y_pack = torch.zeros(y_elems, dtype=torch.bfloat16, device=dev)
        gen = synth.normal_bf16((x_elems,), synth.X_STD, seed=seed + 12345, device=dev)
        self.x_pack.copy_(gen)
        xo = yo = 0
        for (N, K, M) in cases:
            R = self.weights[(N, K)].shape[0]
            xs = self.x_pack[xo:xo + R * M * K].view(R, M, K)
            ys = self.y_pack[yo:yo + R * M * N].view(R, M, N)
            xo += R * M * K
            yo += R * M * N
            plan = sk.sgemm_plan_select(N, K, M)
            self.cases.append({"N": N, "K": K, "M": M, "R": R, "x": xs, "y": ys, "plan": plan,
                               "graphs": {}})
        self.x_host = torch.empty(x_elems, dtype=torch.bfloat16, pin_memory=True)
        self.y_host = torch.empty(y_elems, dtype=torch.bfloat16, pin_memory=True)
        self.x_host.copy_(self.x_pack.cpu())

    def launches_per_step(self):
        return sum(c["R"] * (2 if c["plan"].split_k > 1 else 1) for c in self.cases)

    def capture(self, flags_list):
        """One graph per (case, launch flags); the GEMMs go through the public
        sgemm_bf16_skinny_ex call with the selected plan."""
        torch, sk = self.torch, self.sk
        for c in self.cases:  # eager pass first (allocates split-K scratch outside capture)
            W = self.weights[(c["N"], c["K"])]
            for i in range(c["R"]):
                sk.sgemm_bf16_skinny_ex(c["x"][i], W[i], c["y"][i], plan=c["plan"])
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        for flags in flags_list:
            for c in self.cases:
                W = self.weights[(c["N"], c["K"])]
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        for i in range(c["R"]):
                            sk.sgemm_bf16_skinny_ex(c["x"][i], W[i], c["y"][i], plan=c["plan"],
                                                    flags=flags)
                c["graphs"][flags] = g
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def bytes_per_step(self):
        return sum(c["R"] * gemm_bytes(c["M"], c["N"], c["K"]) for c in self.cases)

    def run_step(self, flags, events=None):
        for j, c in enumerate(self.cases):
            c["graphs"][flags].replay()
            if events is not None:
                events[j + 1].record()


def time_steps(torch, dist, gs, steps, warmup, flags, e2e=False, sampler=None):
    """Run warm-up then exactly `steps` timed steps; returns (max-over-ranks
    seconds, per-case per-step durations in ms)."""
    nc = len(gs.cases)

    def one(events=None):
        if e2e:  # the step's inputs come from pinned host memory, its outputs go back
            gs.x_pack.copy_(gs.x_host, non_blocking=True)
        gs.run_step(flags, events)
        if e2e:
            gs.y_host.copy_(gs.y_pack, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    per_case = [[] for _ in range(nc)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nc + 1)] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    start.record()
    for i in range(steps):
        if e2e:
            one()
        else:
            ev[i][0].record()
            one(ev[i])
    stop.record()
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop() if sampler else None
    total_s = start.elapsed_time(stop) / 1e3
    if not e2e:
        for i in range(steps):
            for j in range(nc):
                per_case[j].append(ev[i][j].elapsed_time(ev[i][j + 1]))
    return dist.max(total_s), per_case, clocks


def cpu_baseline(gs_cases, budget_s=12.0, reference_rows=None):
    """Time the CPU oracle on a bounded sample of the workload: the first rows
    of every (N, K, M) GEMM, sized to about `budget_s` seconds."""
    import oracle
    from bf16_skinny_gemm_gb300 import synth

    threads = oracle.cores()
    cases = [(c["N"], c["K"], c["M"]) for c in gs_cases]
    max_rows = 4096
    inputs = {}
    for (N, K, M) in cases:
        if (N, K) not in inputs:
            inputs[(N, K)] = synth.bits(synth.normal_bf16((min(N, max_rows), K), synth.W_STD,
                                                          seed=0))
    xs = {(K, M): synth.bits(synth.normal_bf16((M, K), 1.0, seed=M)) for (_, K, M) in cases}

    def run(rows):
        t0 = time.perf_counter()
        nbytes = 0
        for (N, K, M) in cases:
            r = min(rows, N)
            _, used = oracle.skinny_gemm(xs[(K, M)], inputs[(N, K)][:r], threads=threads,
                                         return_threads=True)
            nbytes += gemm_bytes(M, r, K)
        return time.perf_counter() - t0, nbytes, used

    if reference_rows is None:
        t, _, _ = run(16)
        rows = min(max_rows, max(16, int(16 * budget_s / max(t, 1e-3))))
    else:
        rows = reference_rows
    t, nbytes, used = run(rows)
    return {"value": nbytes / t / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": f"first {rows} rows of W for each of the {len(cases)} (N,K,M) GEMMs of "
                      f"the step (all M rows of x), {t:.1f} s on {used} threads; "
                      f"throughput scales linearly in rows"}, rows


def reference_arm(args):
    """The oracle as the reference implementation: each step a bounded sample
    of the sweep workload on the host cores."""
    import oracle
    from bf16_skinny_gemm_gb300 import synth

    ws, rank, _ = dist_info()
    if rank != 0:
        return 0
    cases = [(N, K, M) for (N, K) in SWEEP_SHAPES for M in SWEEP_MS]
    rows = args.reference_rows
    W = {(N, K): synth.bits(synth.normal_bf16((min(rows, N), K), synth.W_STD, seed=0))
         for (N, K) in SWEEP_SHAPES}
    X = {(K, M): synth.bits(synth.normal_bf16((M, K), 1.0, seed=M)) for (_, K, M) in cases}
    threads = oracle.cores()

    def step():
        nb = 0
        used = threads
        for (N, K, M) in cases:
            _, used = oracle.skinny_gemm(X[(K, M)], W[(N, K)], threads=threads, return_threads=True)
            nb += gemm_bytes(M, min(rows, N), K)
        return nb, used

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    nb = 0
    for _ in range(args.steps):
        b, used = step()
        nb += b
    t = time.perf_counter() - t0
    v = nb / t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": sweep_config_desc(None),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": used,
                             "kind": "oracle",
                             "sample": f"each step: the first {rows} W rows of each of the 18 "
                                       f"(N,K,M) sweep GEMMs, all M rows of x"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def sweep_config_desc(gs):
    d = {"workload": "shape sweep at M=1,2,4 over local (N,K) = " +
                     ", ".join(f"({N},{K})" for N, K in SWEEP_SHAPES),
         "x": "BF16 ~ N(0,1)", "W": "BF16 ~ N(0,0.02^2)", "seed": 0,
         "l2": "inputs larger than L2: each GEMM reads its own weight copy; copies per shape "
               "total >= max(1 GiB, 4 x L2)",
         "timing": "CUDA graph per (N,K,M) of R GEMMs on R copies; CUDA events per graph",
         "launch": "sgemm_bf16_skinny_ex with the selected plan; the timed chains use the launch "
                   "flags in 'launch_flags' (weights are never written inside the chain)",
         "parallelism": "replicas"}
    if gs is not None:
        d["copies"] = {f"{c['N']}x{c['K']}": c["R"] for c in gs.cases if c["M"] == 1}
    return d


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["sweep", "single", "lmhead", "pairs", "chain"],
                    default="sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--min-bytes", type=float, default=float(1 << 30),
                    help="weight bytes per (N,K) rotation set (at least 4 x L2 is enforced)")
    ap.add_argument("--reference-rows", type=int, default=32)
    ap.add_argument("--shapes", default=None,
                    help="override the sweep shapes, e.g. 12576x4096,4096x1024 (profiling runs)")
    ap.add_argument("--ms", default=None, help="override the sweep M values, e.g. 1,4")
    ap.add_argument("--flags", default="pdl,readonly",
                    help="launch flags of the timed chains: comma list of pdl, readonly, or none")
    ap.add_argument("--no-plain", action="store_true",
                    help="skip the extra timing of plain launches (no launch flags)")
    ap.add_argument("--detail-out", default=None, help="also write the full result JSON here")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.impl == "reference":
        return reference_arm(args)

    import torch

    ws, rank, local = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    torch.cuda.set_device(local)
    dist = Dist(torch)

    import bf16_skinny_gemm_gb300 as sk
    from bf16_skinny_gemm_gb300 import synth

    sk.load()
    sk.sgemm_init()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    min_bytes = max(args.min_bytes, 4 * l2)

    if args.workload == "sweep":
        shapes = SWEEP_SHAPES
        if args.shapes:
            shapes = [tuple(int(v) for v in t.split("x")) for t in args.shapes.split(",")]
        ms = [int(v) for v in args.ms.split(",")] if args.ms else SWEEP_MS
        cases = [(N, K, M) for (N, K) in shapes for M in ms]
    elif args.workload == "single":
        cases = [(4096, 1024, 1)]
    elif args.workload == "lmhead":
        cases = [(LMHEAD[0], LMHEAD[1], M) for M in SWEEP_MS]
    else:
        raise SystemExit(f"workload {args.workload!r} is not available yet")

    flags = 0
    for f in args.flags.split(","):
        flags |= {"pdl": sk.SGEMM_FLAG_PDL, "readonly": sk.SGEMM_FLAG_WEIGHTS_READONLY,
                  "none": 0}[f.strip()]
    flag_sets = [flags] if (args.no_plain or flags == 0) else [flags, 0]
    gs = GraphSet(torch, sk, synth, cases, min_bytes, seed=0)
    gs.capture(flag_sets)
    peak, peak_src = measured_peaks()

    sampler = ClockSampler(local) if rank == 0 else None
    total_s, per_case, clocks = time_steps(torch, dist, gs, args.steps, args.warmup, flags,
                                           sampler=sampler)
    plain_case = None
    if len(flag_sets) > 1:
        _, plain_case, _ = time_steps(torch, dist, gs, args.steps, args.warmup, 0)
    step_bytes = gs.bytes_per_step()
    all_bytes = dist.sum(step_bytes * args.steps)
    value = all_bytes / total_s / 1e9

    detail, kern_bytes, kern_ms = [], 0, 0.0
    traffic, traffic_src = recorded_traffic()
    traffic_sum, traffic_cnt = 0.0, 0
    for ci, (c, ms) in enumerate(zip(gs.cases, per_case)):
        med = statistics.median(ms)
        us = med * 1e3 / c["R"]
        b = gemm_bytes(c["M"], c["N"], c["K"])
        extra = {}
        if plain_case is not None:
            us_plain = statistics.median(plain_case[ci]) * 1e3 / c["R"]
            extra = {"us_plain_launch": round(us_plain, 3),
                     "gbs_plain_launch": round(b / us_plain / 1e3, 1)}
        detail.append({"N": c["N"], "K": c["K"], "M": c["M"], "copies": c["R"],
                       "us": round(us, 3), "gbs": round(b / us / 1e3, 1),
                       "frac": round(b / us / 1e3 / peak, 4), **extra,
                       "plan": {k: v for k, v in c["plan"].as_dict().items()
                                if k in ("threads", "rows_per_warp", "lanes_per_row", "k_unroll",
                                         "split_k", "id")}})
        kern_bytes += c["R"] * b * len(ms)
        kern_ms += sum(ms)
        key = (c["N"], c["K"], c["M"])
        if key in traffic:
            traffic_sum += traffic[key]
            traffic_cnt += 1
    for d in detail:
        base = [e for e in detail if e["N"] == d["N"] and e["K"] == d["K"] and e["M"] == 1]
        if base:
            d["time_vs_m1"] = round(d["us"] / base[0]["us"], 3)
    n_launch = gs.launches_per_step() * args.steps
    achieved = kern_bytes / (kern_ms / 1e3) / 1e9
    launches_timed = sum(c["R"] for c in gs.cases) * args.steps
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (copy bandwidth)",
                "traffic": (round(traffic_sum / traffic_cnt) if traffic_cnt == len(gs.cases)
                            else None),
                "traffic_note": ("mean DRAM bytes per launch over the (N,K,M) cases, from ncu"
                                 if traffic_cnt == len(gs.cases) else traffic_src),
                "algorithmic_bytes_per_launch": round(kern_bytes / launches_timed)}

    e2e = None
    if not args.no_e2e:
        e2e_s, _, _ = time_steps(torch, dist, gs, args.steps, args.warmup, flags, e2e=True)
        e2e = {"value": round(all_bytes / e2e_s / 1e9, 1), "unit": "GB/s",
               "h2d_bytes_per_step": gs.x_host.numel() * 2,
               "d2h_bytes_per_step": gs.y_host.numel() * 2}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu, _ = cpu_baseline(gs.cases)
        cpu["value"] = round(cpu["value"], 4)

    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_s / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(sweep_config_desc(gs), launch_flags=args.flags) if args.workload == "sweep" else
            {"workload": f"{args.workload}: " + ", ".join(f"M={m} ({n},{k})" for n, k, m in cases),
             "l2": "inputs larger than L2 (rotating weight copies)", "parallelism": "replicas"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n_launch,
            "clocks": clocks, "detail": detail}
    if rank == 0:
        print(json.dumps(line), flush=True)
        if args.detail_out:
            with open(args.detail_out, "w") as f:
                json.dump(line, f, indent=1)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
