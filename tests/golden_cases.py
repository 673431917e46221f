"""Parser for the hand-derived fixtures in ``tests/golden/``."""
from __future__ import annotations

import os
from dataclasses import dataclass

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@dataclass
class Case:
    name: str
    why: str
    M: int
    N: int
    K: int
    x: np.ndarray      # uint16 [M, K]
    W: np.ndarray      # uint16 [N, K]
    y: np.ndarray      # uint16 [M, N]
    y_nan: np.ndarray  # bool [M, N]: expected NaN


def _words(tokens):
    out = []
    for t in tokens:
        if "*" in t:
            h, n = t.split("*")
            out.extend([int(h, 16)] * int(n))
        else:
            out.append(int(t, 16))
    return out


def load(filename: str = "closed_forms.txt") -> list[Case]:
    cases, cur = [], {}
    with open(os.path.join(GOLDEN_DIR, filename)) as f:
        lines = [ln.strip() for ln in f] + [""]
    for ln in lines:
        if ln.startswith("#"):
            continue
        if not ln:
            if cur:
                M, N, K = cur["shape"]
                ytok = cur["y"]
                nan = np.array([t == "nan" for t in ytok]).reshape(M, N)
                yv = np.array([0 if t == "nan" else int(t, 16) for t in ytok],
                              dtype=np.uint16).reshape(M, N)
                x = np.array(_words(cur["x"]), dtype=np.uint16)
                W = np.array(_words(cur["W"]), dtype=np.uint16)
                assert x.size == M * K and W.size == N * K and yv.size == M * N, cur["case"]
                cases.append(Case(cur["case"], cur.get("why", ""), M, N, K,
                                  x.reshape(M, K), W.reshape(N, K), yv, nan))
                cur = {}
            continue
        key, _, rest = ln.partition(" ")
        rest = rest.strip()
        if key == "case":
            cur["case"] = rest
        elif key == "why":
            cur["why"] = rest
        elif key == "shape":
            cur["shape"] = tuple(int(v) for v in rest.split())
        elif key in ("x", "W", "y"):
            cur[key] = rest.split()
        else:
            raise ValueError(f"bad fixture line: {ln!r}")
    return cases
