"""Cold-L2 benchmark of the GB300 BF16 skinny GEMM.

Default workload (one "step"): the decode-shape sweep at M = 1, 2, 4 over the
local (N, K) shapes (12576,4096), (4096,4096), (2048,4096), (4096,1024),
(8192,1536), (4096,8192), plus the LM head (77440,4096) at M = 1, 2, 4.
Following the measurement protocol of vLLM PR
#65306 (Validation: each case is a chain over copies of the weight adding up to
at least 1 GiB, captured in a CUDA graph) and PR #62949 (Validation: cold-L2
numbers, the weight rotated out of L2), every (shape, M) is a CUDA graph of R
GEMMs, each on its own weight copy, with R copies totalling
>= max(1 GiB, 4 x L2).  So every GEMM reads its weights from HBM.

Reported on rank 0: a compact table (per shape: us per GEMM, fraction of the
HBM peak and time relative to M=1, at each M; then the paired projection and
the decode chain, timed after the step) followed by one JSON line:
- value: algorithmic bytes (W + x + y) of the whole step / device time, GB/s,
  summed over ranks (replicas: each GPU runs the whole sweep);
- detail (only in the --detail-out file): per (N, K, M) cold-L2 us per GEMM,
  GB/s, fraction of HBM peak, the plan, and the pairs and chain results;
- roofline: the skinny kernel's achieved GB/s against the measured HBM peak;
- e2e: the same metric with every step's x copied in from pinned host memory
  and every y copied back, through the library's public call;
- cpu_baseline: the CPU oracle timed on a bounded sample on this host.

``--impl reference`` times the CPU oracle alone (the reference arm).
``--workload`` selects other configurations: single, lmhead, pairs, chain (with
the elementwise step separate and fused into the GEMM epilogue), router (the
FP32-output router gate), wide (M = 5..8, with cuBLAS timed beside for context).
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
import threading
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
ROUTER = (288, 4096)
CHAIN = [((12576, 4096), 34), ((4096, 4096), 34), ((2048, 4096), 53), ((4096, 1024), 42),
         ((8192, 1536), 11), ((4096, 8192), 11), ((77440, 4096), 1)]
FALLBACK_HBM_GBS = 6800.0


def gemm_bytes(M, N, K):
    """Algorithmic bytes of one GEMM: W + x + y, BF16."""
    return 2 * (N * K + M * K + M * N)


def launches_per_gemm(sk, plan):
    """Kernel launches of one GEMM: split-K plans of the streaming and 16-row
    tensor-core kernels add a second-pass reduce; the tcgen05 kernel and the
    cluster-split streaming plans reduce their K split inside a cluster."""
    one_launch = (sk.SGEMM_VARIANT_TC05, sk.SGEMM_VARIANT_LDG_CLUSTER)
    return 2 if plan.split_k > 1 and plan.variant not in one_launch else 1


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


# The streaming kernels' sources, their compiled configurations, the plan table and
# the launch geometry: what the recorded DRAM traffic per launch depends on.
KERNEL_SOURCES = ["skinny_ldg.cuh", "skinny_mma.cuh", "skinny_tc05.cuh", "tc05_consts.h", "tc05_launch.cu",
                  "kernel_table.cuh", "internal.h", "plan_table.inc", "api.cpp"]


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bf16_skinny_gemm_gb300", "csrc")
    for name in KERNEL_SOURCES:
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

    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.first = 0
        self.reader = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln)

    def start(self):
        """Start sampling and return once the first sample is in (at most 2 s), so that
        the timed region that follows is sampled from its beginning; samples taken
        before this returns are not counted."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t0 = time.monotonic()
        while not self.lines and time.monotonic() - t0 < 2.0 and self.proc.poll() is None:
            time.sleep(0.005)
        self.first = len(self.lines)

    def stop(self):
        if self.proc is None:
            return None
        n_in_region = len(self.lines)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.reader.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.first:n_in_region]:
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
        return sum(c["R"] * launches_per_gemm(self.sk, c["plan"]) for c in self.cases)

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
    shapes = list(SWEEP_SHAPES) + ([] if args.no_lmhead else [LMHEAD])
    cases = [(N, K, M) for (N, K) in shapes for M in SWEEP_MS]
    rows = args.reference_rows
    W = {(N, K): synth.bits(synth.normal_bf16((min(rows, N), K), synth.W_STD, seed=0))
         for (N, K) in shapes}
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
            "config": dict(sweep_config_desc(None, lmhead=not args.no_lmhead),
                           launch_flags=args.flags),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": used,
                             "kind": "oracle",
                             "sample": f"each step: the first {rows} W rows of each of the "
                                       f"{len(cases)} (N,K,M) GEMMs of the step, all M rows of x"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _time_graphs(torch, dist, graphs, steps, warmup):
    """Replay each graph `warmup` then `steps` times; per-graph median ms and the
    max-over-ranks total seconds of the timed replays."""
    for _ in range(warmup):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
          for _ in range(steps)]
    dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(steps):
        ev[i][0].record()
        for j, g in enumerate(graphs):
            g.replay()
            ev[i][j + 1].record()
    stop.record()
    torch.cuda.synchronize()
    dist.barrier()
    per = [statistics.median(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
           for j in range(len(graphs))]
    return per, dist.max(start.elapsed_time(stop) / 1e3)


def _capture(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def pairs_result(args, torch, sk, synth, dist, min_bytes):
    """Paired projection f_b / g_b, (N, K) = (4096, 128), M = 1..4: both problems
    in ONE batched launch, against two separate launches of the same kernel
    (vLLM PR #57617, Microbenchmark table: two Linear calls vs one paired call).
    Weights rotate through copies totalling >= 4 x L2 (cold)."""
    ws, rank, _ = dist_info()
    N, K = PAIR
    dev = torch.device("cuda")
    R = max(2, math.ceil(min_bytes / (2 * 2 * N * K)))
    W = torch.empty((R, 2, N, K), dtype=torch.bfloat16, device=dev)
    for i in range(R):
        for j in range(2):
            W[i, j].copy_(synth.normal_bf16((N, K), synth.PAIR_W_STD, seed=2 * i + j, device=dev))
    flags = sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY
    # every buffer a captured graph uses must outlive the graph: entering a graph
    # capture empties the allocator cache, so a freed buffer would be unmapped
    detail, graphs, nbytes, keep = [], [], 0, []
    for M in SWEEP_MS + [3]:
        x = synth.normal_bf16((R, 2, M, K), synth.X_STD, seed=100 + M, device=dev)
        y = torch.empty((R, 2, M, N), dtype=torch.bfloat16, device=dev)
        keep.append((x, y))

        def paired():
            for i in range(R):
                sk.sgemm_bf16_skinny_batched_ex([(x[i, 0], W[i, 0], y[i, 0]),
                                                 (x[i, 1], W[i, 1], y[i, 1])], flags=flags)

        def separate():
            for i in range(R):
                for j in range(2):
                    sk.sgemm_bf16_skinny_ex(x[i, j], W[i, j], y[i, j], flags=flags)

        paired()
        separate()
        torch.cuda.synchronize()
        graphs += [_capture(torch, paired), _capture(torch, separate)]
        detail.append({"M": M, "copies": R})
        nbytes += R * 2 * gemm_bytes(M, N, K)
    per, _ = _time_graphs(torch, dist, graphs, args.steps, args.warmup)
    del graphs, keep
    total_ms = 0.0
    for d, (p_ms, s_ms) in zip(detail, zip(per[0::2], per[1::2])):
        d["us_per_paired_launch"] = round(p_ms * 1e3 / d["copies"], 3)
        d["us_two_launches"] = round(s_ms * 1e3 / d["copies"], 3)
        b = 2 * gemm_bytes(d["M"], N, K)
        d["gbs_paired"] = round(b / (p_ms * 1e3 / d["copies"]) / 1e3, 1)
        total_ms += p_ms
    value = dist.sum(nbytes) / (dist.max(total_ms) / 1e3) / 1e9
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "paired batched projection f_b/g_b: batch 2 x (N,K)=(4096,128), "
                                   "M=1..4, one launch for both",
                       "x": "BF16 ~ N(0,1)", "W": "BF16 ~ N(0,0.05^2)",
                       "l2": "inputs larger than L2 (rotating weight copies)",
                       "launch_flags": "pdl,readonly", "parallelism": "replicas"},
            "gpu_launches": sum(d["copies"] * 3 for d in detail) * args.steps,
            "detail": detail}
    return line


def chain_result(args, torch, sk, synth, dist):
    """Decode-step chain at M=1: 186 GEMMs on distinct weights in the order
    (12576,4096)x34, (4096,4096)x34, (2048,4096)x53, (4096,1024)x42,
    (8192,1536)x11, (4096,8192)x11, (77440,4096)x1 (7.5 GB of weights, so every
    GEMM is cold), each output fed through the elementwise rescale kernel into
    the next GEMM's input, the whole step one CUDA graph.  The elementwise
    kernels are also timed alone and subtracted (as vLLM PR #65306 does)."""
    ws, rank, _ = dist_info()
    dev = torch.device("cuda")
    seq = [shape for shape, count in CHAIN for _ in range(count)]
    Ws = [synth.normal_bf16(shape, synth.W_STD, seed=i, device=dev) for i, shape in enumerate(seq)]
    xs = [torch.empty((1, K), dtype=torch.bfloat16, device=dev) for (_, K) in seq]
    ys = [torch.empty((1, N), dtype=torch.bfloat16, device=dev) for (N, _) in seq]
    xs[0].copy_(synth.normal_bf16((1, seq[0][1]), synth.X_STD, seed=999, device=dev))
    scales = [1.0 / (synth.W_STD * math.sqrt(K)) for (_, K) in seq]
    flags = sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY
    if args.flags == "none":
        flags = 0

    def step():
        for i in range(len(seq)):
            sk.sgemm_bf16_skinny_ex(xs[i], Ws[i], ys[i], flags=flags)
            if i + 1 < len(seq):
                sk.sgemm_bf16_rescale(ys[i], xs[i + 1], scales[i], flags=flags & sk.SGEMM_FLAG_PDL)

    def elementwise_only():
        for i in range(len(seq) - 1):
            sk.sgemm_bf16_rescale(ys[i], xs[i + 1], scales[i], flags=flags & sk.SGEMM_FLAG_PDL)

    def fused_step():
        # the elementwise step in each GEMM's epilogue: 186 launches instead of 371
        for i in range(len(seq)):
            if i + 1 < len(seq):
                sk.sgemm_bf16_skinny_rescale_ex(xs[i], Ws[i], ys[i], xs[i + 1], scales[i],
                                                flags=flags)
            else:
                sk.sgemm_bf16_skinny_ex(xs[i], Ws[i], ys[i], flags=flags)

    step()
    torch.cuda.synchronize()
    y_last = ys[-1].clone()
    fused_step()
    torch.cuda.synchronize()
    if not torch.equal(ys[-1].view(torch.int16), y_last.view(torch.int16)):
        raise SystemExit("fused chain step differs from the separate one")
    g_step = _capture(torch, step)
    g_elt = _capture(torch, elementwise_only)
    g_fused = _capture(torch, fused_step)
    per, total_s = _time_graphs(torch, dist, [g_step, g_elt, g_fused], args.steps, args.warmup)
    step_ms, elt_ms, fused_ms = per
    w_bytes = sum(2 * N * K for (N, K) in seq)
    alg = sum(gemm_bytes(1, N, K) for (N, K) in seq)
    gemm_ms = step_ms - elt_ms
    peak, src = measured_peaks()
    value = dist.sum(alg) / (dist.max(gemm_ms) / 1e3) / 1e9
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "decode-step chain at M=1, 186 GEMMs on distinct weights, "
                                   "elementwise rescale between GEMMs, one CUDA graph",
                       "weights_bytes": w_bytes, "l2": "inputs larger than L2 (7.5 GB of "
                       "distinct weights per step)", "launch_flags": args.flags,
                       "parallelism": "replicas"},
            "chain": {"step_us": round(step_ms * 1e3, 1),
                      "elementwise_us": round(elt_ms * 1e3, 1),
                      "gemm_us": round(gemm_ms * 1e3, 1),
                      "gemm_us_at_measured_peak": round(alg / (peak * 1e9) * 1e6, 1),
                      "frac_of_peak": round(alg / (gemm_ms / 1e3) / 1e9 / peak, 4),
                      "peak_source": src,
                      "fused_step_us": round(fused_ms * 1e3, 1),
                      "fused_gbs": round(alg / (fused_ms / 1e3) / 1e9, 1),
                      "fused_frac_of_peak": round(alg / (fused_ms / 1e3) / 1e9 / peak, 4),
                      "fused_note": "the same chain with the elementwise step in each GEMM's "
                                    "epilogue (sgemm_bf16_skinny_rescale_ex), whole step, "
                                    "nothing subtracted; outputs bitwise equal"},
            "gpu_launches": ((2 * len(seq) - 1) + (len(seq) - 1) + len(seq)) * args.steps}
    return line


def emit(line, args, dist):
    """Print the JSON line on rank 0 (and write it to --detail-out), then close."""
    if dist_info()[1] == 0:
        print(json.dumps(line), flush=True)
        if args.detail_out:
            with open(args.detail_out, "w") as f:
                json.dump(line, f, indent=1)
    dist.close()
    return 0


def run_pairs(args, torch, sk, synth, dist, min_bytes):
    return emit(pairs_result(args, torch, sk, synth, dist, min_bytes), args, dist)


def run_chain(args, torch, sk, synth, dist):
    return emit(chain_result(args, torch, sk, synth, dist), args, dist)


def sweep_config_desc(gs, lmhead=True):
    d = {"workload": "shape sweep at M=1,2,4 over local (N,K) = " +
                     ", ".join(f"({N},{K})" for N, K in SWEEP_SHAPES) +
                     (" and the LM head (77440,4096)" if lmhead else ""),
         "x": "BF16 ~ N(0,1)", "W": "BF16 ~ N(0,0.02^2)", "seed": 0,
         "l2": "inputs larger than L2: each GEMM reads its own weight copy, copies per shape "
               ">= max(1 GiB, 4 x L2)",
         "timing": "a CUDA graph of R GEMMs per (N,K,M); CUDA events",
         "parallelism": "replicas"}
    return d


def compact_table(detail, peak, extras):
    """Short per-shape lines for stdout: us per GEMM, fraction of the HBM peak
    and time relative to M=1, at each M."""
    lines = [f"# cold-L2 us per GEMM / fraction of {peak:.0f} GB/s / time vs M=1 (plan variant)"]
    shapes = []
    for d in detail:
        if (d["N"], d["K"]) not in shapes:
            shapes.append((d["N"], d["K"]))
    for (N, K) in shapes:
        row = [d for d in detail if d["N"] == N and d["K"] == K]
        cells = " ".join(f"M{d['M']} {d['us']:.2f}/{d['frac']:.3f}/{d.get('time_vs_m1', 1.0):.2f}"
                         f"(v{d['plan']['variant']})" for d in row)
        lines.append(f"# {N}x{K} {cells}")
    for e in extras:
        lines.append("# " + e)
    return lines


def run_router(args, torch, sk, synth, dist, min_bytes):
    """The MoE router gate (N, K) = (288, 4096) with FP32 outputs, M = 1..4, the
    projection vLLM PR #62949 (Validation, the nsys census) leaves on cuBLAS for
    its FP32 output.  Each M: a CUDA graph of R GEMMs on R weight copies (cold),
    FP32 outputs (sgemm_bf16_skinny_f32out_ex) and, for comparison, BF16 outputs."""
    ws, rank, _ = dist_info()
    N, K = ROUTER
    dev = torch.device("cuda")
    R = max(2, math.ceil(min_bytes / (2 * N * K)))
    W = torch.empty((R, N, K), dtype=torch.bfloat16, device=dev)
    for i in range(R):
        W[i].copy_(synth.normal_bf16((N, K), synth.W_STD, seed=i, device=dev))
    flags = sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY
    detail, graphs, keep, nbytes = [], [], [], 0
    for M in [1, 2, 3, 4]:
        x = synth.normal_bf16((R, M, K), synth.X_STD, seed=200 + M, device=dev)
        y32 = torch.empty((R, M, N), dtype=torch.float32, device=dev)
        y16 = torch.empty((R, M, N), dtype=torch.bfloat16, device=dev)
        keep.append((x, y32, y16))

        def f32():
            for i in range(R):
                sk.sgemm_bf16_skinny_f32out_ex(x[i], W[i], y32[i], flags=flags)

        def b16():
            for i in range(R):
                sk.sgemm_bf16_skinny_ex(x[i], W[i], y16[i], flags=flags)

        f32()
        b16()
        torch.cuda.synchronize()
        graphs += [_capture(torch, f32), _capture(torch, b16)]
        detail.append({"M": M, "copies": R})
        nbytes += R * (2 * (N * K + M * K) + 4 * M * N)
    per, _ = _time_graphs(torch, dist, graphs, args.steps, args.warmup)
    del graphs, keep
    total_ms = 0.0
    for d, (f_ms, b_ms) in zip(detail, zip(per[0::2], per[1::2])):
        d["us_f32_out"] = round(f_ms * 1e3 / d["copies"], 3)
        d["us_bf16_out"] = round(b_ms * 1e3 / d["copies"], 3)
        d["gbs_f32_out"] = round((2 * (N * K + d["M"] * K) + 4 * d["M"] * N)
                                 / (f_ms * 1e3 / d["copies"]) / 1e3, 1)
        total_ms += f_ms
    value = dist.sum(nbytes) / (dist.max(total_ms) / 1e3) / 1e9
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "router gate (N,K)=(288,4096), FP32 outputs, M=1..4",
                       "x": "BF16 ~ N(0,1)", "W": "BF16 ~ N(0,0.02^2)",
                       "l2": "inputs larger than L2 (rotating weight copies)",
                       "launch_flags": "pdl,readonly", "parallelism": "replicas"},
            "gpu_launches": sum(d["copies"] * 2 for d in detail) * args.steps,
            "detail": detail}
    if rank == 0:
        print(json.dumps(line), flush=True)
        if args.detail_out:
            with open(args.detail_out, "w") as f:
                json.dump(line, f, indent=1)
    dist.close()
    return 0


def run_wide(args, torch, sk, synth, dist, min_bytes):
    """Wider batches, M = 5..8 (speculative verification), over the sweep shapes:
    each (N, K, M) a CUDA graph of R GEMMs on R weight copies (cold), through
    sgemm_bf16_skinny_ex with the selected plan.  For context only, the same
    graphs through torch's F.linear (cuBLAS), which is where vLLM PR #62949
    (Validation) leaves M = 8; nothing of this library runs in that column."""
    import torch.nn.functional as F
    ws, rank, _ = dist_info()
    dev = torch.device("cuda")
    flags = sk.SGEMM_FLAG_PDL | sk.SGEMM_FLAG_WEIGHTS_READONLY
    ms = [int(v) for v in args.ms.split(",")] if args.ms else [5, 6, 7, 8]
    shapes = SWEEP_SHAPES
    if args.shapes:
        shapes = [tuple(int(v) for v in t.split("x")) for t in args.shapes.split(",")]
    detail, graphs, keep, nbytes, launches = [], [], [], 0, 0
    for (N, K) in shapes:
        R = max(2, math.ceil(min_bytes / (2 * N * K)))
        W = torch.empty((R, N, K), dtype=torch.bfloat16, device=dev)
        for i in range(R):
            W[i].copy_(synth.normal_bf16((N, K), synth.W_STD, seed=i, device=dev))
        for M in ms:
            x = synth.normal_bf16((R, M, K), synth.X_STD, seed=300 + M, device=dev)
            y = torch.empty((R, M, N), dtype=torch.bfloat16, device=dev)
            yc = torch.empty((R, M, N), dtype=torch.bfloat16, device=dev)
            keep.append((W, x, y, yc))

            def ours(W=W, x=x, y=y, R=R):
                for i in range(R):
                    sk.sgemm_bf16_skinny_ex(x[i], W[i], y[i], flags=flags)

            def cublas(W=W, x=x, yc=yc, R=R):
                for i in range(R):
                    torch.matmul(x[i], W[i].T, out=yc[i])

            ours()
            cublas()
            torch.cuda.synchronize()
            graphs += [_capture(torch, ours), _capture(torch, cublas)]
            p = sk.sgemm_plan_select(N, K, M)
            detail.append({"N": N, "K": K, "M": M, "copies": R,
                           "plan": {"variant": p.variant, "threads": p.threads,
                                    "k_unroll": p.k_unroll, "split_k": p.split_k, "id": p.id}})
            nbytes += R * gemm_bytes(M, N, K)
            launches += R * launches_per_gemm(sk, p)
    per, _ = _time_graphs(torch, dist, graphs, args.steps, args.warmup)
    del graphs, keep
    peak, _ = measured_peaks()
    total_ms = 0.0
    for d, (o_ms, c_ms) in zip(detail, zip(per[0::2], per[1::2])):
        b = gemm_bytes(d["M"], d["N"], d["K"])
        d["us"] = round(o_ms * 1e3 / d["copies"], 3)
        d["gbs"] = round(b / (o_ms * 1e3 / d["copies"]) / 1e3, 1)
        d["frac"] = round(d["gbs"] / peak, 4)
        d["us_cublas_informational"] = round(c_ms * 1e3 / d["copies"], 3)
        total_ms += o_ms
    value = dist.sum(nbytes) / (dist.max(total_ms) / 1e3) / 1e9
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "wide batches M=" + ",".join(map(str, ms)) + " over (N,K) = " +
                                   ", ".join(f"({n},{k})" for n, k in shapes),
                       "x": "BF16 ~ N(0,1)", "W": "BF16 ~ N(0,0.02^2)",
                       "l2": "inputs larger than L2 (rotating weight copies)",
                       "launch_flags": "pdl,readonly", "parallelism": "replicas"},
            "gpu_launches": launches * args.steps,
            "detail": detail}
    if rank == 0:
        print(json.dumps(line), flush=True)
        if args.detail_out:
            with open(args.detail_out, "w") as f:
                json.dump(line, f, indent=1)
    dist.close()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload",
                    choices=["sweep", "single", "lmhead", "pairs", "chain", "router", "wide"],
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
    ap.add_argument("--no-lmhead", action="store_true",
                    help="leave the LM head (77440,4096) out of the default step")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the paired-projection and decode-chain lines after the step")
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
        shapes = list(SWEEP_SHAPES)
        if not args.no_lmhead:
            shapes.append(LMHEAD)
        if args.shapes:
            shapes = [tuple(int(v) for v in t.split("x")) for t in args.shapes.split(",")]
        ms = [int(v) for v in args.ms.split(",")] if args.ms else SWEEP_MS
        cases = [(N, K, M) for (N, K) in shapes for M in ms]
    elif args.workload == "single":
        cases = [(4096, 1024, 1)]
    elif args.workload == "lmhead":
        cases = [(LMHEAD[0], LMHEAD[1], M) for M in SWEEP_MS]
    elif args.workload == "pairs":
        return run_pairs(args, torch, sk, synth, dist, min_bytes)
    elif args.workload == "router":
        return run_router(args, torch, sk, synth, dist, min_bytes)
    elif args.workload == "wide":
        return run_wide(args, torch, sk, synth, dist, min_bytes)
    else:
        return run_chain(args, torch, sk, synth, dist)

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
                       "plan": c["plan"].as_dict()})
        kern_bytes += c["R"] * b * len(ms)
        kern_ms += sum(ms)
        key = (c["N"], c["K"], c["M"])
        if key in traffic:  # weighted like the achieved bytes: by launches in the step
            traffic_sum += traffic[key] * c["R"]
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
                "traffic": (round(traffic_sum / sum(c["R"] for c in gs.cases))
                            if traffic_cnt == len(gs.cases) else None),
                "traffic_note": ("DRAM bytes per launch of the step (ncu, per case, weighted by "
                                 "launches like 'achieved')"
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

    # the paired projection and the decode chain, timed after the step (not in value)
    extras, extra_detail = [], {}
    if args.workload == "sweep" and not args.no_extras:
        pr = pairs_result(args, torch, sk, synth, dist, min_bytes)
        extra_detail["pairs"] = pr
        extras.append("pairs 2x(4096,128) us/launch " + " ".join(
            f"M{d['M']} {d['us_per_paired_launch']:.2f}" for d in pr["detail"]) +
            " (two launches: " + " ".join(f"{d['us_two_launches']:.2f}" for d in pr["detail"]) + ")")
        ch = chain_result(args, torch, sk, synth, dist)
        extra_detail["chain"] = ch
        c = ch["chain"]
        extras.append(f"chain 186 GEMMs M=1: fused step {c['fused_step_us']:.0f} us "
                      f"({c['fused_frac_of_peak']:.3f} of peak), separate {c['step_us']:.0f} us, "
                      f"GEMMs alone {c['gemm_us']:.0f} us ({c['frac_of_peak']:.3f})")

    config = (sweep_config_desc(gs, lmhead=LMHEAD in [(c["N"], c["K"]) for c in gs.cases])
              if args.workload == "sweep" else
              {"workload": f"{args.workload}: " + ", ".join(f"M={m} ({n},{k})" for n, k, m in cases),
               "l2": "inputs larger than L2 (rotating weight copies)", "parallelism": "replicas"})
    config["launch_flags"] = args.flags
    roofline.pop("traffic_note", None)
    if cpu is not None:
        cpu["sample"] = cpu["sample"].split(";")[0]
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_s / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": n_launch, "clocks": clocks}
    if rank == 0:
        for ln in compact_table(detail, peak, extras):
            print(ln, flush=True)
        print(json.dumps(line), flush=True)
        if args.detail_out:
            with open(args.detail_out, "w") as f:
                json.dump(dict(line, detail=detail, traffic_source=traffic_src, **extra_detail),
                          f, indent=1)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
