"""Pins for the oracle's other element types: bfloat16 and binary16 operands, and FP64.

As for FP32, nothing here re-types the oracle's loop: the 16-bit widenings are checked
against hand-derived encodings and the ordering of the formats, and the FP64 product against
exact integer and dyadic arithmetic, hand-derived binary64 rounding cases, a closed form and
the standard inner-product error bound. Planted mistakes in copies of the source must fail a
pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

import oracle
from golden_io import bf16_values, rounding_cases
from roofline_driven_tiling_gb300 import inputs

MODES = (oracle.MUL_ADD, oracle.FMA)
U64 = 2.0 ** -53  # unit roundoff of binary64


def gamma64(k: int) -> float:
    """gamma_k for binary64 (Higham, Accuracy and Stability of Numerical Algorithms, 2nd ed.,
    eq. 3.5 with lemma 3.1)."""
    return k * U64 / (1.0 - k * U64)


# ----------------------------------------------------------------------------------------
# bfloat16 widening and the bfloat16 product
# ----------------------------------------------------------------------------------------

def check_bf16_encodings(o):
    """Hand-derived encodings decode to their values (sign, zero, subnormal, inf, NaN)."""
    table = bf16_values()
    bits = np.array([b for b, _ in table], dtype=np.uint16)
    got = o.bf16_to_f32(bits)
    for (b, want), g in zip(table, got):
        g = float(g)
        if math.isnan(want):
            if not math.isnan(g):
                return False, "0x%04X: %r is not NaN" % (b, g)
        elif g != want or math.copysign(1.0, g) != math.copysign(1.0, want):
            return False, "0x%04X: %r != %r" % (b, g, want)
    return True, ""


def check_bf16_order_and_sign(o):
    """Over all 65536 patterns: the non-negative finite ones increase strictly with the
    pattern (IEEE sign-magnitude encoding), and setting the sign bit negates."""
    pos = np.arange(0x0000, 0x7F81, dtype=np.uint16)  # +0 .. +inf
    v = o.bf16_to_f32(pos).astype(np.float64)
    if not np.all(np.diff(v) > 0):
        return False, "positive patterns are not strictly increasing"
    neg = o.bf16_to_f32(pos | np.uint16(0x8000)).astype(np.float64)
    if not np.array_equal(neg, -v) or not np.all(np.signbit(neg)):
        return False, "the sign bit does not negate"
    nan = o.bf16_to_f32(np.arange(0x7F81, 0x8000, dtype=np.uint16))
    if not np.all(np.isnan(nan)):
        return False, "exponent 255 with a fraction must be NaN"
    return True, ""


def check_bf16_product_exact(o):
    """Integer-pattern and small dyadic operands in bfloat16: exact, so C equals the exact
    product bit for bit (int64 / float64 matmul, exact for these inputs)."""
    for (M, N, K) in [(19, 23, 45), (64, 8, 130)]:
        A, B = inputs.integer_pattern(M, N, K)
        exact = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
        C = o.gemm_bf16(inputs.to_bf16_bits(A), inputs.to_bf16_bits(B))
        if not np.array_equal(C.view(np.uint32), exact.view(np.uint32)):
            return False, "bf16 integer pattern %s" % ((M, N, K),)
    A = inputs.dyadic(17, 40, seed=5, denom=16, span=64)  # |j| <= 64: 7 bits, exact in bf16
    B = inputs.dyadic(40, 9, seed=6, denom=16, span=64)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    C = o.gemm_bf16(inputs.to_bf16_bits(A), inputs.to_bf16_bits(B))
    if not np.array_equal(C.astype(np.float64), exact):
        return False, "bf16 dyadic"
    return True, ""


def check_bf16_random_bound(o):
    """Random bfloat16 operands: within gamma_K (binary32) of the exact sum, elementwise."""
    for t, (M, N, K) in enumerate([(9, 7, 33), (16, 5, 200)]):
        Ab = inputs.uniform_bf16(M, K, 700 + t)
        Bb = inputs.uniform_bf16(K, N, 800 + t)
        A, B = o.bf16_to_f32(Ab).astype(np.float64), o.bf16_to_f32(Bb).astype(np.float64)
        exact = A @ B
        absb = np.abs(A) @ np.abs(B)
        C = o.gemm_bf16(Ab, Bb).astype(np.float64)
        g = K * 2.0 ** -24 / (1 - K * 2.0 ** -24)
        if np.any(np.abs(C - exact) > g * absb):
            return False, "bf16 error bound %s" % ((M, N, K),)
    return True, ""


BF16_BATTERY = [check_bf16_encodings, check_bf16_order_and_sign, check_bf16_product_exact,
                check_bf16_random_bound]


# ----------------------------------------------------------------------------------------
# IEEE binary16 widening and the binary16 product
# ----------------------------------------------------------------------------------------

def check_f16_encodings(o):
    """Hand-derived binary16 encodings decode to their values (subnormals included)."""
    table = bf16_values("f16_values.txt")
    got = o.f16_to_f32(np.array([b for b, _ in table], dtype=np.uint16))
    for (b, want), g in zip(table, got):
        g = float(g)
        if math.isnan(want):
            if not math.isnan(g):
                return False, "0x%04X: %r is not NaN" % (b, g)
        elif g != want or math.copysign(1.0, g) != math.copysign(1.0, want):
            return False, "0x%04X: %r != %r" % (b, g, want)
    return True, ""


def check_f16_order_and_sign(o):
    """Over all patterns: +0 .. +inf increase strictly with the pattern, the subnormals are
    evenly spaced by 2^-24, the sign bit negates, exponent 31 with a fraction is NaN."""
    pos = np.arange(0x0000, 0x7C01, dtype=np.uint16)
    v = o.f16_to_f32(pos).astype(np.float64)
    if not np.all(np.diff(v) > 0):
        return False, "positive patterns are not strictly increasing"
    if not np.array_equal(v[:0x401], np.arange(0x401) * 2.0 ** -24):
        return False, "subnormals and the first normal are not multiples of 2^-24"
    neg = o.f16_to_f32(pos | np.uint16(0x8000)).astype(np.float64)
    if not np.array_equal(neg, -v) or not np.all(np.signbit(neg)):
        return False, "the sign bit does not negate"
    if not np.all(np.isnan(o.f16_to_f32(np.arange(0x7C01, 0x8000, dtype=np.uint16)))):
        return False, "exponent 31 with a fraction must be NaN"
    return True, ""


def check_f16_product_exact(o):
    """Integer-pattern and 11-bit dyadic operands in binary16: C equals the exact product."""
    for (M, N, K) in [(19, 23, 45), (64, 8, 130)]:
        A, B = inputs.integer_pattern(M, N, K)
        exact = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
        C = o.gemm_f16(inputs.to_f16_bits(A), inputs.to_f16_bits(B))
        if not np.array_equal(C.view(np.uint32), exact.view(np.uint32)):
            return False, "f16 integer pattern %s" % ((M, N, K),)
    A = inputs.dyadic(17, 40, seed=15, denom=256, span=1000)  # |j| <= 1000: exact in binary16
    B = inputs.dyadic(40, 9, seed=16, denom=16, span=64)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    C = o.gemm_f16(inputs.to_f16_bits(A), inputs.to_f16_bits(B))
    if not np.array_equal(C.astype(np.float64), exact):
        return False, "f16 dyadic"
    return True, ""


def check_f16_random_bound(o):
    """Random binary16 operands: within gamma_K (binary32) of the exact sum, elementwise."""
    for t, (M, N, K) in enumerate([(9, 7, 33), (16, 5, 200)]):
        Ab = inputs.uniform_f16(M, K, 720 + t)
        Bb = inputs.uniform_f16(K, N, 820 + t)
        A, B = o.f16_to_f32(Ab).astype(np.float64), o.f16_to_f32(Bb).astype(np.float64)
        C = o.gemm_f16(Ab, Bb).astype(np.float64)
        g = K * 2.0 ** -24 / (1 - K * 2.0 ** -24)
        if np.any(np.abs(C - A @ B) > g * (np.abs(A) @ np.abs(B))):
            return False, "f16 error bound %s" % ((M, N, K),)
    return True, ""


F16_BATTERY = [check_f16_encodings, check_f16_order_and_sign, check_f16_product_exact,
               check_f16_random_bound]


# ----------------------------------------------------------------------------------------
# FP64
# ----------------------------------------------------------------------------------------

def check_f64_integer_exact(o):
    """Integer-pattern inputs: every FP64 step is exact, so C equals the int64 product."""
    for (M, N, K) in [(33, 20, 71), (5, 40, 3)]:
        A, B = inputs.integer_pattern(M, N, K)
        exact = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64)
        for mode in MODES:
            C = o.dgemm(A.astype(np.float64), B.astype(np.float64), mode)
            if not np.array_equal(C, exact):
                return False, "f64 integer pattern %s mode %d" % ((M, N, K), mode)
    return True, ""


def check_f64_rounding_cases(o):
    """Hand-derived binary64 cases that separate the two modes and fix ascending k."""
    for name, A, B, c_mul_add, c_fma in rounding_cases("rounding_cases_f64.txt", np.float64):
        for mode, want in ((oracle.MUL_ADD, c_mul_add), (oracle.FMA, c_fma)):
            C = o.dgemm(A, B, mode)
            if not np.array_equal(C.view(np.uint64), want.view(np.uint64)):
                return False, "%s mode %d: %r != %r" % (name, mode, C, want)
    return True, ""


def check_f64_constant_closed_form(o, n: int = 40, k: int = 300):
    """A = 0.5, B = 0.4: every entry is one number within gamma_K * K * |a b| of 0.2 K."""
    A = np.full((n, k), 0.5)
    B = np.full((k, n + 3), 0.4)
    exact = k * 0.5 * 0.4
    for mode in MODES:
        C = o.dgemm(A, B, mode)
        if not np.all(C == C[0, 0]):
            return False, "constant inputs gave unequal entries (mode %d)" % mode
        if abs(float(C[0, 0]) - exact) > gamma64(k) * exact:
            return False, "constant: %r vs %r" % (float(C[0, 0]), exact)
    return True, ""


def check_f64_random_bound(o):
    """Uniform binary64 inputs: |C - exact| <= gamma_K (|A| |B|), with the exact sum taken in
    rationals on small shapes; and FP64 rounding is actually seen."""
    from fractions import Fraction
    saw_rounding = False
    for t, (M, N, K) in enumerate([(3, 4, 17), (2, 3, 64)]):
        A = inputs.uniform_f64(M, K, 900 + t)
        B = inputs.uniform_f64(K, N, 950 + t)
        for mode in MODES:
            C = o.dgemm(A, B, mode)
            for i in range(M):
                for j in range(N):
                    ex = sum(Fraction(A[i, k]) * Fraction(B[k, j]) for k in range(K))
                    absb = sum(abs(A[i, k] * B[k, j]) for k in range(K))
                    err = abs(Fraction(C[i, j]) - ex)
                    if err > Fraction(gamma64(K) * absb):
                        return False, "f64 error bound %s mode %d" % ((M, N, K), mode)
                    saw_rounding |= err != 0
    if not saw_rounding:
        return False, "no FP64 rounding seen: the accumulator is wider than binary64"
    return True, ""


def check_f64_sampled_and_empty(o):
    """The sampled entry agrees with the full product; K = 0 gives +0.0."""
    A = inputs.uniform_f64(21, 13, 3)
    B = inputs.uniform_f64(13, 17, 4)
    rng = np.random.default_rng(1)
    rows, cols = rng.integers(0, 21, 100), rng.integers(0, 17, 100)
    for mode in MODES:
        C = o.dgemm(A, B, mode)
        if not np.array_equal(o.dgemm_at(A, B, rows, cols, mode).view(np.uint64),
                              C[rows, cols].view(np.uint64)):
            return False, "sampled entries differ (mode %d)" % mode
        Z = o.dgemm(np.zeros((3, 0)), np.zeros((0, 4)), mode)
        if Z.shape != (3, 4) or np.any(Z.view(np.uint64) != 0):
            return False, "K = 0 must give +0.0"
    return True, ""


F64_BATTERY = [check_f64_integer_exact, check_f64_rounding_cases, check_f64_constant_closed_form,
               check_f64_random_bound, check_f64_sampled_and_empty]


@pytest.mark.parametrize("check", BF16_BATTERY + F16_BATTERY + F64_BATTERY,
                         ids=[c.__name__ for c in BF16_BATTERY + F16_BATTERY + F64_BATTERY])
def test_oracle_type_pin(check):
    ok, detail = check(oracle.default())
    assert ok, detail


def test_type_entries_reject_bad_arguments():
    o = oracle.default()
    with pytest.raises(TypeError):
        o.bf16_to_f32(np.zeros(3, np.int16))
    with pytest.raises(TypeError):
        o.dgemm(np.zeros((2, 2), np.float32), np.zeros((2, 2), np.float32))
    with pytest.raises(ValueError):
        o.dgemm_at(np.zeros((2, 2)), np.zeros((2, 2)), [2], [0])
    with pytest.raises(ValueError):
        inputs.to_bf16_bits(np.array([1.0 + 2.0 ** -10], np.float32))
    with pytest.raises(TypeError):
        o.f16_to_f32(np.zeros(3, np.float16))
    with pytest.raises(ValueError):
        inputs.to_f16_bits(np.array([1.0 + 2.0 ** -12], np.float32))


# ----------------------------------------------------------------------------------------
# Planted mistakes
# ----------------------------------------------------------------------------------------

MUTANTS = {
    # bfloat16 widening
    "bf16_shift_15": ("(uint32_t)x[i] << 16", "(uint32_t)x[i] << 15"),
    "bf16_sign_dropped": ("(uint32_t)x[i] << 16", "(uint32_t)(x[i] & 0x7fffu) << 16"),
    "bf16_low_half_set": ("(uint32_t)x[i] << 16", "((uint32_t)x[i] << 16) | 0x8000u"),
    "bf16_byte_swapped": ("(uint32_t)x[i] << 16",
                          "(uint32_t)(uint16_t)((x[i] >> 8) | (x[i] << 8)) << 16"),
    # binary16 widening
    "f16_wrong_bias": ("ldexp(1.0 + (double)f / 1024.0, e - 15)", "ldexp(1.0 + (double)f / 1024.0, e - 16)"),
    "f16_subnormal_as_normal": ("v = ldexp((double)f, -24);", "v = ldexp(1.0 + (double)f / 1024.0, -14);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "f16_fraction_bits": ("const unsigned f = x[i] & 0x3ffu;", "const unsigned f = x[i] & 0x1ffu;"),
    "f16_sign_dropped": ("y[i] = (float)(sign ? -v : v);", "y[i] = (float)v;"),
    "f16_no_infinity": ("v = f == 0 ? INFINITY : NAN;", "v = ldexp(1.0 + (double)f / 1024.0, 16);"),
    # FP64 product
    "f64_transposed_B": ("const double b = B[k * N + j];", "const double b = B[j * K + k];"),
    "f64_reversed_k_in_A": ("const double a = A[i * K + k];",
                            "const double a = A[i * K + (K - 1 - k)];"),
    "f64_nonzero_start": ("double acc = 0.0;", "double acc = 1.0;"),
    "f64_float_accumulator": ("double acc = 0.0;", "float acc = 0.0f;"),
    "f64_wide_accumulator": ("double acc = 0.0;", "long double acc = 0.0L;"),
    "f64_unfused_in_fma_mode": ("acc = fma(a, b, acc);", "acc = acc + a * b;"),
    "f64_fused_in_mul_add_mode": ("const double p = a * b; /* rounded to FP64 here */",
                                  "const double p = 0.0; acc = fma(a, b, acc);"),
    "f64_wrong_sign": ("acc = acc + p;          /* and rounded again here */",
                       "acc = acc - p;          /* and rounded again here */"),
    "f64_descending_k": ("for (int64_t k = 0; k < K; ++k) {\n        const double a",
                         "for (int64_t k = K - 1; k >= 0; --k) {\n        const double a"),
    "f64_dropped_last_term": ("for (int64_t k = 0; k < K; ++k) {\n        const double a",
                              "for (int64_t k = 0; k < K - 1; ++k) {\n        const double a"),
    "f64_transposed_C": ("C[i * N + j] = dot_row_col_f64", "C[j * M + i] = dot_row_col_f64"),
}


@pytest.fixture(scope="module")
def oracle_source():
    with open(os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c"), encoding="utf-8") as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_type_mistake_is_caught(name, oracle_source, tmp_path):
    old, new = MUTANTS[name]
    assert oracle_source.count(old) == 1, "mutation site missing or not unique: %r" % old
    src = tmp_path / ("mutant_%s.c" % name)
    src.write_text(oracle_source.replace(old, new), encoding="utf-8")
    lib = oracle.compile_source(str(src), str(tmp_path / ("libmutant_%s.so" % name)))
    mutant = oracle.Oracle(lib)
    battery = (BF16_BATTERY if name.startswith("bf16") else
               F16_BATTERY if name.startswith("f16") else F64_BATTERY)
    failed = [c.__name__ for c in battery if not c(mutant)[0]]
    assert failed, "planted mistake %r passed every pin" % name
