"""Seeded synthetic inputs for the FP32 GEMM workloads.

This module only makes input matrices; it holds none of the multiply's
arithmetic, so both the CUDA path's tests and the CPU oracle's tests draw their
inputs from here without sharing any computation.

Three input kinds, each a row-major float32 array:

* ``integer_pattern`` -- A[i] = (i % 13) - 6 over the flat index of A and
  B[i] = (i % 7) - 3 over the flat index of B (page "GEMM 커널 테스트 코드 작성
  및 최적화 (1024^3 크기 실험)", section "Host 코드와 타이밍 방식", the
  "데이터 초기화" loops). Every product is an integer of magnitude at most 18 and
  every partial sum of K terms is at most 18*K in magnitude, so for K < 2**24/18
  every FP32 operation on them is exact.
* ``constant`` -- A filled with 0.5 and B with 0.4 (page "[AutoMine++] #2. 행렬
  곱셈 구현 시행착오", section "직관적 구현 (by CPU)", the ``main`` that times
  the CPU loop).
* ``uniform`` -- i.i.d. values on [-1, 1). The pages give no generator, so this
  module defines one: a counter-based SplitMix64 stream (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014; the output
  function of Vigna's reference ``splitmix64.c``). Output s of seed ``seed`` is
  ``mix(seed + (s + 1) * 0x9E3779B97F4A7C15)`` (mod 2**64), and the float is
  ``(u >> 40) * 2**-23 - 1``: an exact 2**24-point grid on [-1, 1), so the value
  does not depend on any rounding.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

#: Seeds of the uniform workloads: A uses 1000 + config number, B 2000 + config number.
SEED_A_BASE = 1000
SEED_B_BASE = 2000


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream with the given seed (uint64)."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + ctr * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform(rows: int, cols: int, seed: int) -> np.ndarray:
    """rows x cols float32 matrix, i.i.d. on the 2**-23 grid of [-1, 1)."""
    n = int(rows) * int(cols)
    out = np.empty(n, dtype=np.float32)
    chunk = 1 << 24
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        u = splitmix64(seed, e - s, start=s)
        hi = (u >> np.uint64(40)).astype(np.int64)  # 24 random bits
        out[s:e] = (hi.astype(np.float64) * 2.0 ** -23 - 1.0).astype(np.float32)
    return out.reshape(rows, cols)


def integer_pattern(M: int, N: int, K: int):
    """(A, B) with A[i] = (i % 13) - 6 and B[i] = (i % 7) - 3 over flat indices."""
    a = (np.arange(M * K, dtype=np.int64) % 13 - 6).astype(np.float32).reshape(M, K)
    b = (np.arange(K * N, dtype=np.int64) % 7 - 3).astype(np.float32).reshape(K, N)
    return a, b


def constant(M: int, N: int, K: int, a: float = 0.5, b: float = 0.4):
    """(A, B) filled with the constants a and b (as float32)."""
    return (np.full((M, K), a, dtype=np.float32), np.full((K, N), b, dtype=np.float32))


def uniform_pair(M: int, N: int, K: int, config_no: int):
    """(A, B) uniform on [-1, 1) with the seeds 1000 + config_no and 2000 + config_no."""
    return (uniform(M, K, SEED_A_BASE + config_no), uniform(K, N, SEED_B_BASE + config_no))


def dyadic(rows: int, cols: int, seed: int, denom: int = 16, span: int = 32) -> np.ndarray:
    """Small dyadic rationals j/denom with |j| <= span, drawn from the same stream.

    Products and short sums of such values are exact in FP32, so a product of
    small dyadic matrices has one exact answer that any order of summation reaches.
    """
    u = splitmix64(seed, rows * cols)
    j = (u % np.uint64(2 * span + 1)).astype(np.int64) - span
    return (j.astype(np.float64) / denom).astype(np.float32).reshape(rows, cols)


def uniform_f64(rows: int, cols: int, seed: int) -> np.ndarray:
    """rows x cols float64 matrix, i.i.d. on the 2**-52 grid of [-1, 1): output s of the
    stream gives ``(u >> 11) * 2**-52 - 1`` (53 random bits, exact in binary64)."""
    n = int(rows) * int(cols)
    out = np.empty(n, dtype=np.float64)
    chunk = 1 << 24
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        u = splitmix64(seed, e - s, start=s)
        hi = (u >> np.uint64(11)).astype(np.int64)  # 53 random bits, < 2**53
        out[s:e] = hi.astype(np.float64) * 2.0 ** -52 - 1.0
    return out.reshape(rows, cols)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bfloat16 bit patterns of float32 values that bfloat16 holds exactly (the upper
    half of each binary32 encoding). Raises ValueError for a value bfloat16 cannot hold."""
    v = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if np.any(v & np.uint32(0xFFFF)):
        raise ValueError("a value is not representable in bfloat16")
    return (v >> np.uint32(16)).astype(np.uint16)


def uniform_bf16(rows: int, cols: int, seed: int) -> np.ndarray:
    """rows x cols bfloat16 bit patterns: the ``uniform`` values with the low 16 bits of each
    binary32 encoding cleared (the value moved toward zero onto the bfloat16 grid)."""
    v = uniform(rows, cols, seed).view(np.uint32)
    return (v >> np.uint32(16)).astype(np.uint16)


def uniform_f16(rows: int, cols: int, seed: int) -> np.ndarray:
    """rows x cols IEEE binary16 bit patterns, i.i.d. on the 2**-11 grid of [-1, 1): output s
    of the stream gives ``((u >> 52) - 2048) / 2048`` (12 random bits; every such value has
    at most 11 significant bits and is exact in binary16, so the conversion does not round)."""
    u = splitmix64(seed, int(rows) * int(cols))
    j = (u >> np.uint64(52)).astype(np.int64) - 2048
    return (j.astype(np.float64) / 2048.0).astype(np.float16).view(np.uint16).reshape(rows, cols)


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 binary16 bit patterns of float32 values that binary16 holds exactly. Raises
    ValueError for a value binary16 cannot hold."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    h = x.astype(np.float16)
    if not np.array_equal(h.astype(np.float32), x, equal_nan=True):
        raise ValueError("a value is not representable in binary16")
    return h.view(np.uint16)


# The workloads: (name, M, N, K, kind, config number).
CONFIGS = {
    "c1_int_256": (256, 256, 256, "integer", 1),
    "c2_int_1024": (1024, 1024, 1024, "integer", 2),
    "c2_const_1024": (1024, 1024, 1024, "constant", 2),
    "c3_ragged": (1000, 1003, 997, "uniform", 3),
    "c4_uniform_4096": (4096, 4096, 4096, "uniform", 4),
}

#: Roofline sweep shapes (M, N, K), uniform inputs, config number 5.
SWEEP = [(n, n, n) for n in (128, 256, 512, 1024, 2048, 4096, 8192)] + [
    (16384, 16384, 32), (8192, 8192, 64)]


def make(kind: str, M: int, N: int, K: int, config_no: int):
    """Inputs of one kind for an M x N x K product."""
    if kind == "integer":
        return integer_pattern(M, N, K)
    if kind == "constant":
        return constant(M, N, K)
    if kind == "uniform":
        return uniform_pair(M, N, K, config_no)
    raise ValueError("unknown input kind %r" % kind)
