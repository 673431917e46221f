"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The skinny GEMM runs on one GPU per call: bench.py runs one
independent replica per GPU (no collective on the data path).  What crosses
ranks is only the timing protocol: a barrier around the timed region, the MAX
of the elapsed times and the SUM of the bytes processed, and rank 0 alone
printing.  These tests run that logic with two gloo ranks.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch

    import bench

    d = bench.Dist(torch, backend="gloo")
    d.barrier()
    elapsed = 1.0 + rank          # rank 1 is the slow one
    nbytes = 100.0 * (rank + 1)
    q.put((rank, d.max(elapsed), d.sum(nbytes)))
    d.barrier()
    d.close()


def test_max_time_and_sum_bytes_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tmax, bsum in res:
        assert tmax == 2.0, "elapsed time must be the max over ranks"
        assert bsum == 300.0, "bytes must be summed over ranks"


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2",
           "--warmup", "3", "--reference-rows", "8"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_bench_rejects_short_warmup():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


@pytest.mark.parametrize("M,N,K,expect", [(1, 4096, 1024, 8398848), (4, 12576, 4096, 103155968)])
def test_algorithmic_bytes(M, N, K, expect):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.gemm_bytes(M, N, K) == expect


def test_clock_sampler_counts_only_the_timed_region(tmp_path, monkeypatch):
    """The bench's nvidia-smi sampler, against a fake nvidia-smi on PATH: samples
    before start() returns are not counted, throttle reasons are collected."""
    import time

    sys.path.insert(0, ROOT)
    import bench

    fake = tmp_path / "nvidia-smi"
    fake.write_text(
        "#!/bin/bash\n"
        "echo '0, 1000, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
        "while true; do\n"
        "  echo '0, 2070, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active'\n"
        "  sleep 0.02\n"
        "done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}:{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(0.2)
    c = s.stop()
    assert c is not None and c["samples"] >= 3
    assert c["sm_mhz"] == 2070.0  # the 1000 MHz line came before start() returned
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("PATH", str(tmp_path))
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop() is None
