"""The cache-blocked multi-core CPU GEMM (the stronger CPU baseline) against the oracle.

It sums every element by fused multiply-adds in ascending k from +0.0f, blocked over i, j and
k chunks for cache reuse, so it must equal the oracle's fused-multiply-add reading bit for bit
on every input: the edges of every blocking level (ragged M, N and K around MR, NR, MC, NC and
KC), several K chunks, empty shapes and special values. It is a baseline only; it checks
nothing itself.
"""
from __future__ import annotations

import numpy as np
import pytest

import cpu_baseline
import oracle
from roofline_driven_tiling_gb300 import inputs


def bits_equal(x, y):
    return np.array_equal(x.view(np.uint32), y.view(np.uint32))


@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 15, 3), (6, 16, 256), (7, 17, 257),
                                   (95, 255, 511), (97, 257, 513), (200, 300, 700),
                                   (193, 520, 1030)],
                         ids=lambda s: "x".join(map(str, s)))
def test_blocked_equals_fma_oracle(shape):
    M, N, K = shape
    A, B = inputs.uniform_pair(M, N, K, 31)
    got = cpu_baseline.sgemm(A, B)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert bits_equal(got, want)


def test_blocked_integer_pattern_exact():
    A, B = inputs.integer_pattern(256, 256, 256)
    exact = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
    assert bits_equal(cpu_baseline.sgemm(A, B), exact)


def test_blocked_special_values_and_empty_shapes():
    M, N, K = 37, 41, 300
    A, B = inputs.uniform_pair(M, N, K, 32)
    A[3, 5], A[7, 299], B[0, 2], B[150, 40] = np.nan, np.inf, -np.inf, np.float32(1e-45)
    got = cpu_baseline.sgemm(A, B)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert bits_equal(got[ok], want[ok])
    assert cpu_baseline.sgemm(np.zeros((0, 4), np.float32), np.zeros((4, 3), np.float32)).shape == (0, 3)
    z = cpu_baseline.sgemm(np.zeros((3, 0), np.float32), np.zeros((0, 5), np.float32))
    assert z.shape == (3, 5) and bits_equal(z, np.zeros((3, 5), np.float32))


def test_blocked_thread_count_does_not_change_bits():
    A, B = inputs.uniform_pair(150, 170, 600, 33)
    n = cpu_baseline.num_threads()
    try:
        cpu_baseline.set_num_threads(1)
        one = cpu_baseline.sgemm(A, B)
    finally:
        cpu_baseline.set_num_threads(n)
    assert bits_equal(one, cpu_baseline.sgemm(A, B))
