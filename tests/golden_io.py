"""Readers for the text fixtures under tests/golden/."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def page_figures() -> dict:
    """name -> float from page_figures.txt (the citation column is dropped)."""
    out = {}
    with open(os.path.join(GOLDEN, "page_figures.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head = line.split("|", 1)[0]
            name, value = (t.strip() for t in head.split("=", 1))
            out[name] = float(value)
    return out


def rounding_cases() -> list:
    """[(name, A, B, C_mul_add, C_fma)] from rounding_cases.txt, as float32 arrays."""
    cases = []
    with open(os.path.join(GOLDEN, "rounding_cases.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, dims, a, b, c0, c1 = (t.strip() for t in line.split("|"))
            M, N, K = (int(t) for t in dims.split())
            A = np.array([float.fromhex(t) for t in a.split()], dtype=np.float32).reshape(M, K)
            B = np.array([float.fromhex(t) for t in b.split()], dtype=np.float32).reshape(K, N)
            C0 = np.array([float.fromhex(t) for t in c0.split()], dtype=np.float32).reshape(M, N)
            C1 = np.array([float.fromhex(t) for t in c1.split()], dtype=np.float32).reshape(M, N)
            cases.append((name, A, B, C0, C1))
    return cases
