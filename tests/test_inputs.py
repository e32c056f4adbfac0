"""Pins of the seeded input generator (no GPU).

The uniform workloads are drawn from a SplitMix64 stream. These tests tie the generator to
the published outputs of the reference SplitMix64 (tests/golden/splitmix64.txt) and check the
stated map from 64-bit outputs to floats on [-1, 1), so that every uniform-input parity case
and bench workload is the stream its description says it is.
"""
from __future__ import annotations

import os

import numpy as np

from roofline_driven_tiling_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "splitmix64.txt")


def published_outputs():
    rows = []
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            seed, idx, out = (t.strip() for t in line.split("|"))
            rows.append((int(seed), int(idx), int(out, 16)))
    return rows


def test_splitmix64_matches_published_outputs():
    rows = published_outputs()
    assert len(rows) >= 3
    for seed, idx, want in rows:
        got = int(inputs.splitmix64(seed, 1, start=idx)[0])
        assert got == want, "seed %d call %d: %#x vs %#x" % (seed, idx, got, want)


def test_splitmix64_stream_offsets_are_consistent():
    whole = inputs.splitmix64(1004, 1000)
    for start in (0, 1, 17, 999):
        part = inputs.splitmix64(1004, 1000 - start, start=start)
        assert np.array_equal(part, whole[start:])


def test_uniform_is_the_stated_map_of_the_stream():
    """x = (u >> 40) * 2^-23 - 1, computed here in exact integer arithmetic: 24 random bits on
    a 2^24-point grid of [-1, 1), every value exact in binary32."""
    rows, cols, seed = 7, 13, 1003
    got = inputs.uniform(rows, cols, seed).ravel()
    u = inputs.splitmix64(seed, rows * cols)
    for x, w in zip(got, u):
        hi = int(w) >> 40
        want = (hi - (1 << 23)) / float(1 << 23)
        assert float(x) == want
    assert np.all(got >= -1.0) and np.all(got < 1.0)


def test_uniform_seeds_differ_between_operands():
    A = inputs.uniform(64, 64, inputs.SEED_A_BASE + 3)
    B = inputs.uniform(64, 64, inputs.SEED_B_BASE + 3)
    assert not np.array_equal(A, B)
    # Near-uniform use of the grid: the mean of 4096 values is within a few sigma of 0.
    assert abs(float(A.mean())) < 4 * (1 / np.sqrt(3)) / 64
