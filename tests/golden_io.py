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


def rounding_cases(fname: str = "rounding_cases.txt", dtype=np.float32) -> list:
    """[(name, A, B, C_mul_add, C_fma)] from a rounding-case fixture, as arrays of `dtype`."""
    cases = []
    with open(os.path.join(GOLDEN, fname), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, dims, a, b, c0, c1 = (t.strip() for t in line.split("|"))
            M, N, K = (int(t) for t in dims.split())
            A = np.array([float.fromhex(t) for t in a.split()], dtype=dtype).reshape(M, K)
            B = np.array([float.fromhex(t) for t in b.split()], dtype=dtype).reshape(K, N)
            C0 = np.array([float.fromhex(t) for t in c0.split()], dtype=dtype).reshape(M, N)
            C1 = np.array([float.fromhex(t) for t in c1.split()], dtype=dtype).reshape(M, N)
            cases.append((name, A, B, C0, C1))
    return cases


def bf16_values(fname: str = "bf16_values.txt") -> list:
    """[(bits, value)] from a 16-bit encoding fixture (bf16_values.txt, f16_values.txt); value
    is a Python float (inf / nan included)."""
    out = []
    with open(os.path.join(GOLDEN, fname), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, value, _ = (t.strip() for t in line.split("|", 2))
            v = {"inf": float("inf"), "-inf": float("-inf"), "nan": float("nan")}.get(value)
            out.append((int(bits, 16), float.fromhex(value) if v is None else v))
    return out
