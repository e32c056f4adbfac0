"""Pins for the CPU oracle: checks against what the pages and arithmetic fix.

None of these re-types the oracle's loop. Each compares it with something
independent of it: exact integer or dyadic arithmetic done by numpy's integer /
float64 matmul (a library primitive that is exact for these inputs), closed
forms, a standard error bound, or hand-derived rounding cases. A separate test
plants plausible mistakes in copies of the oracle's source and checks that the
battery catches every one.
"""
from __future__ import annotations

import os
import re
import tempfile

import numpy as np
import pytest

import oracle
from golden_io import page_figures, rounding_cases
from roofline_driven_tiling_gb300 import inputs

MODES = (oracle.MUL_ADD, oracle.FMA)
U = 2.0 ** -24  # unit roundoff of binary32


def gamma(k: int) -> float:
    """gamma_k = k u / (1 - k u): the forward error constant of a k-term inner
    product in floating point (Higham, Accuracy and Stability of Numerical
    Algorithms, 2nd ed., eq. 3.5 with lemma 3.1)."""
    return k * U / (1.0 - k * U)


# ----------------------------------------------------------------------------
# The battery: each check takes an oracle instance and returns (ok, detail).
# ----------------------------------------------------------------------------

def check_integer_pattern_exact(o):
    """Integer-pattern inputs are exact in FP32, so C must equal the int64 product bit for bit."""
    for (M, N, K) in [(64, 64, 64), (37, 29, 53), (5, 40, 3)]:
        A, B = inputs.integer_pattern(M, N, K)
        exact = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
        for mode in MODES:
            C = o.sgemm(A, B, mode)
            if not np.array_equal(C.view(np.uint32), exact.view(np.uint32)):
                return False, "integer pattern %s mode %d" % ((M, N, K), mode)
    return True, ""


def check_dyadic_exact(o):
    """Small dyadic inputs: every partial sum is exact, so C equals the float64 product."""
    shapes = [(1, 1, 1), (3, 5, 7), (17, 1, 33), (1, 19, 4), (33, 31, 2), (8, 9, 10)]
    for t, (M, N, K) in enumerate(shapes):
        A = inputs.dyadic(M, K, seed=11 + t)
        B = inputs.dyadic(K, N, seed=97 + t)
        exact = A.astype(np.float64) @ B.astype(np.float64)
        for mode in MODES:
            C = o.sgemm(A, B, mode)
            if not np.array_equal(C.astype(np.float64), exact):
                return False, "dyadic %s mode %d" % ((M, N, K), mode)
    return True, ""


def check_rounding_cases(o):
    """Hand-derived binary32 cases that separate the two modes and fix ascending k."""
    for name, A, B, c_mul_add, c_fma in rounding_cases():
        for mode, want in ((oracle.MUL_ADD, c_mul_add), (oracle.FMA, c_fma)):
            C = o.sgemm(A, B, mode)
            if not np.array_equal(C.view(np.uint32), want.view(np.uint32)):
                return False, "%s mode %d: %r != %r" % (name, mode, C, want)
    return True, ""


def check_constant_closed_form(o, n: int = 96, k: int = 300):
    """A = 0.5, B = 0.4: every C entry is one number within gamma_K * K * |a b| of 0.2 K."""
    A, B = inputs.constant(n, n + 3, k)
    exact = k * 0.5 * float(np.float32(0.4))  # the exact product for the FP32 inputs
    bound = gamma(k) * k * 0.5 * float(np.float32(0.4))
    for mode in MODES:
        C = o.sgemm(A, B, mode)
        if not np.all(C == C[0, 0]):
            return False, "constant inputs gave unequal entries (mode %d)" % mode
        if abs(float(C[0, 0]) - exact) > bound:
            return False, "constant: %r vs %r (bound %g)" % (float(C[0, 0]), exact, bound)
    return True, ""


def check_error_bound_random(o):
    """Uniform inputs on tiny shapes: |C - C_exact| <= gamma_K * (|A| |B|) elementwise."""
    for t, (M, N, K) in enumerate([(1, 1, 1), (7, 3, 33), (33, 33, 33), (16, 17, 2), (2, 5, 31)]):
        A = inputs.uniform(M, K, 500 + t)
        B = inputs.uniform(K, N, 600 + t)
        exact = A.astype(np.float64) @ B.astype(np.float64)
        absb = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
        for mode in MODES:
            C = o.sgemm(A, B, mode).astype(np.float64)
            if np.any(np.abs(C - exact) > gamma(K) * absb):
                return False, "error bound %s mode %d" % ((M, N, K), mode)
            if K > 1 and np.array_equal(C, exact) and mode == oracle.MUL_ADD and M * N > 50:
                # Random inputs that never round would mean the oracle is not FP32.
                return False, "no FP32 rounding seen %s" % ((M, N, K),)
    return True, ""


def check_sampled_and_rows(o):
    """The element-wise and row-block entries agree with the full product bit for bit."""
    M, N, K = 41, 23, 19
    A = inputs.uniform(M, K, 7)
    B = inputs.uniform(K, N, 8)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, M, 200)
    cols = rng.integers(0, N, 200)
    for mode in MODES:
        C = o.sgemm(A, B, mode)
        at = o.sgemm_at(A, B, rows, cols, mode)
        if not np.array_equal(at.view(np.uint32), C[rows, cols].view(np.uint32)):
            return False, "sampled entries differ (mode %d)" % mode
        blk = o.sgemm_rows(A, B, 5, 17, mode)
        if not np.array_equal(blk.view(np.uint32), C[5:17].view(np.uint32)):
            return False, "row block differs (mode %d)" % mode
    return True, ""


def check_empty(o):
    """K = 0 is the empty sum (+0.0); M = 0 or N = 0 give empty results."""
    for mode in MODES:
        C = o.sgemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32), mode)
        if C.shape != (3, 4) or np.any(C.view(np.uint32) != 0):
            return False, "K = 0 must give +0.0"
        if o.sgemm(np.zeros((0, 5), np.float32), np.zeros((5, 2), np.float32), mode).shape != (0, 2):
            return False, "M = 0"
    return True, ""


BATTERY = [check_integer_pattern_exact, check_dyadic_exact, check_rounding_cases,
           check_constant_closed_form, check_error_bound_random, check_sampled_and_rows,
           check_empty]


@pytest.mark.parametrize("check", BATTERY, ids=[c.__name__ for c in BATTERY])
def test_oracle_pin(check):
    ok, detail = check(oracle.default())
    assert ok, detail


def test_constant_config_closed_form_at_page_size():
    """The page's CPU workload, 1024^3 with A = 0.5 and B = 0.4, against C = 0.2 K."""
    fig = page_figures()
    n = int(fig["cpu_const_n"])
    A, B = inputs.constant(n, n, n, fig["cpu_const_a"], fig["cpu_const_b"])
    exact = n * 0.5 * float(np.float32(0.4))
    assert abs(exact - 0.2 * n) < 1e-5  # 204.8 up to the FP32 rounding of 0.4
    for mode in MODES:
        # The full product is 1e9 multiply-adds; rows 0..63 and the last row suffice to
        # show all entries agree (every row and column holds the same data).
        blk = oracle.sgemm_rows(A, B, 0, 64, mode)
        last = oracle.sgemm_rows(A, B, n - 1, n, mode)
        assert np.all(blk == blk[0, 0]) and np.all(last == blk[0, 0])
        assert abs(float(blk[0, 0]) - exact) <= gamma(n) * exact


def test_integer_pattern_page_size_exact():
    """256^3 integer pattern (the small workload): oracle equals the exact integer product."""
    A, B = inputs.integer_pattern(256, 256, 256)
    exact = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
    for mode in MODES:
        C = oracle.sgemm(A, B, mode)
        assert np.array_equal(C.view(np.uint32), exact.view(np.uint32))
        assert float(np.max(np.abs(C - exact))) == page_figures()["max_abs_diff_naive_vs_tiled"]


def test_oracle_rejects_bad_arguments():
    o = oracle.default()
    with pytest.raises(ValueError):
        o.sgemm(np.zeros((2, 3), np.float32), np.zeros((4, 2), np.float32))
    with pytest.raises(ValueError):
        o.sgemm_at(np.zeros((2, 3), np.float32), np.zeros((3, 2), np.float32), [2], [0])
    with pytest.raises(TypeError):
        o.sgemm(np.zeros((2, 3), np.float64), np.zeros((3, 2), np.float32))


# ----------------------------------------------------------------------------
# Planted mistakes: each is a plausible error in the oracle's source; the battery
# above must reject every one of them.
# ----------------------------------------------------------------------------

MUTANTS = {
    "transposed_B": ("B[k * N + j]", "B[j * K + k]"),
    "A_index_reversed_k": ("A[i * K + k]", "A[i * K + (K - 1 - k)]"),
    "dropped_first_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k < K - 1; ++k)"),
    "descending_k": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = K - 1; k >= 0; --k)"),
    "wrong_sign": ("acc = acc + p;", "acc = acc - p;"),
    "nonzero_start": ("float acc = 0.0f;", "float acc = 1.0f;"),
    "fused_in_mul_add_mode": ("const float p = a * b; /* rounded to FP32 here */",
                              "const float p = 0.0f; acc = fmaf(a, b, acc);"),
    "unfused_in_fma_mode": ("acc = fmaf(a, b, acc);", "acc = acc + a * b;"),
    "double_accumulator": ("float acc = 0.0f;", "double acc = 0.0;"),
    "transposed_C": ("C[i * N + j] = dot_row_col", "C[j * M + i] = dot_row_col"),
    "swapped_operands_in_product": ("const float b = B[k * N + j];", "const float b = B[k * N + (N - 1 - j)];"),
}


@pytest.fixture(scope="module")
def oracle_source():
    with open(os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c"), encoding="utf-8") as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, oracle_source, tmp_path):
    old, new = MUTANTS[name]
    assert oracle_source.count(old) >= 1, "mutation site vanished: %r" % old
    src = tmp_path / ("mutant_%s.c" % name)
    src.write_text(oracle_source.replace(old, new), encoding="utf-8")
    lib = oracle.compile_source(str(src), str(tmp_path / ("libmutant_%s.so" % name)))
    mutant = oracle.Oracle(lib)
    failed = [c.__name__ for c in BATTERY if not c(mutant)[0]]
    assert failed, "planted mistake %r passed every pin" % name


# ----------------------------------------------------------------------------
# Vector add (the memory-roof probe's operation)
# ----------------------------------------------------------------------------

def test_vector_add_exact_and_special():
    o = oracle.default()
    # Dyadic values: every sum is exact, so it equals the float64 sum.
    x = inputs.dyadic(1, 1001, seed=3).ravel()
    y = inputs.dyadic(1, 1001, seed=4).ravel()
    z = o.vector_add(x, y)
    assert np.array_equal(z.astype(np.float64), x.astype(np.float64) + y.astype(np.float64))
    # One rounding: 1 + 2^-24 is a tie and rounds to the even 1.0; 1 + 3 * 2^-24 rounds up.
    z = o.vector_add(np.array([1.0, 1.0], np.float32),
                     np.array([2.0 ** -24, 3 * 2.0 ** -24], np.float32))
    assert z[0] == np.float32(1.0) and z[1] == np.float32(1.0 + 2.0 ** -22)
    z = o.vector_add(np.array([np.inf, -0.0, 3e38], np.float32),
                     np.array([-np.inf, -0.0, 3e38], np.float32))
    assert np.isnan(z[0]) and np.signbit(z[1]) and z[1] == 0 and np.isinf(z[2])
    assert o.vector_add(np.zeros(0, np.float32), np.zeros(0, np.float32)).size == 0
