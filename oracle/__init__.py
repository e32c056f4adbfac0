"""CPU oracle for the row-major FP32 GEMM C = A x B (ctypes loader).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library and
its Python binding never import it, and the product path has no CPU fallback
that could route through it.

The arithmetic lives in ``gemm_oracle.c`` (plain C, FP32 accumulation in
ascending k, built with -ffp-contract=off); this module only compiles it with
gcc and marshals numpy arrays into it. See the header of ``gemm_oracle.c`` for
the definition and the passages of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MUL_ADD = 0  #: acc = fl(acc + fl(a*b)), the C statement with two roundings
FMA = 1  #: acc = fl(acc + a*b), one rounding (fused multiply-add)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_gemm.so")
_CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library at `out` (gcc)."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``liboracle_gemm.so`` (gcc). Returns the path."""
    with _lock:
        stale = (not os.path.exists(_LIB)
                 or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
        if force or stale:
            compile_source(_SRC, _LIB)
    return _LIB


class Oracle:
    """The oracle library at one path (the default build, or a test's variant of it)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, fp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.t2s_oracle_sgemm.argtypes = [i64, i64, i64, fp, fp, fp, ip]
        lib.t2s_oracle_sgemm.restype = ip
        lib.t2s_oracle_sgemm_at.argtypes = [i64, i64, i64, fp, fp, i64, fp, fp, fp, ip]
        lib.t2s_oracle_sgemm_at.restype = ip
        lib.t2s_oracle_sgemm_rows.argtypes = [i64, i64, i64, fp, fp, i64, i64, fp, ip]
        lib.t2s_oracle_sgemm_rows.restype = ip
        lib.t2s_oracle_num_threads.argtypes = []
        lib.t2s_oracle_num_threads.restype = ip
        lib.t2s_oracle_set_num_threads.argtypes = [ip]
        lib.t2s_oracle_set_num_threads.restype = None
        lib.t2s_oracle_vector_add.argtypes = [i64, fp, fp, fp]
        lib.t2s_oracle_vector_add.restype = ip
        lib.t2s_oracle_bf16_to_f32.argtypes = [i64, fp, fp]
        lib.t2s_oracle_bf16_to_f32.restype = ip
        lib.t2s_oracle_f16_to_f32.argtypes = [i64, fp, fp]
        lib.t2s_oracle_f16_to_f32.restype = ip
        lib.t2s_oracle_dgemm.argtypes = [i64, i64, i64, fp, fp, fp, ip]
        lib.t2s_oracle_dgemm.restype = ip
        lib.t2s_oracle_dgemm_at.argtypes = [i64, i64, i64, fp, fp, i64, fp, fp, fp, ip]
        lib.t2s_oracle_dgemm_at.restype = ip
        self.lib = lib

    def vector_add(self, x: np.ndarray, y: np.ndarray) -> np.ndarray:
        """z = x + y elementwise (float32, one rounding per element)."""
        x, y = _f32(x).ravel(), _f32(y).ravel()
        if x.shape != y.shape:
            raise ValueError("x and y differ in length")
        z = np.empty_like(x)
        if self.lib.t2s_oracle_vector_add(x.size, x.ctypes.data, y.ctypes.data, z.ctypes.data) != 0:
            raise ValueError("oracle rejected the arguments")
        return z

    def sgemm(self, A: np.ndarray, B: np.ndarray, mode: int = MUL_ADD) -> np.ndarray:
        """Full product C = A x B (float32, row-major)."""
        A, B = _f32(A), _f32(B)
        M, N, K = _shapes(A, B)
        C = np.empty((M, N), dtype=np.float32)
        rc = self.lib.t2s_oracle_sgemm(M, N, K, A.ctypes.data, B.ctypes.data,
                                       C.ctypes.data, mode)
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return C

    def sgemm_at(self, A: np.ndarray, B: np.ndarray, rows, cols,
                 mode: int = MUL_ADD) -> np.ndarray:
        """Elements C[rows[s], cols[s]] of C = A x B, one by one."""
        A, B = _f32(A), _f32(B)
        M, N, K = _shapes(A, B)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        if rows.shape != cols.shape or rows.ndim != 1:
            raise ValueError("rows and cols must be 1-D and of equal length")
        out = np.empty(rows.shape[0], dtype=np.float32)
        rc = self.lib.t2s_oracle_sgemm_at(M, N, K, A.ctypes.data, B.ctypes.data,
                                          rows.shape[0], rows.ctypes.data,
                                          cols.ctypes.data, out.ctypes.data, mode)
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return out

    def sgemm_rows(self, A: np.ndarray, B: np.ndarray, r0: int, r1: int,
                   mode: int = MUL_ADD) -> np.ndarray:
        """Rows r0..r1-1 of C = A x B."""
        A, B = _f32(A), _f32(B)
        M, N, K = _shapes(A, B)
        out = np.empty((max(r1 - r0, 0), N), dtype=np.float32)
        rc = self.lib.t2s_oracle_sgemm_rows(M, N, K, A.ctypes.data, B.ctypes.data,
                                            r0, r1, out.ctypes.data, mode)
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return out


    def bf16_to_f32(self, bits: np.ndarray) -> np.ndarray:
        """Widen bfloat16 bit patterns (uint16) to the float32 values they encode."""
        bits = np.ascontiguousarray(bits)
        if bits.dtype != np.uint16:
            raise TypeError("bfloat16 inputs must be uint16 bit patterns, got %s" % bits.dtype)
        out = np.empty(bits.shape, dtype=np.float32)
        if self.lib.t2s_oracle_bf16_to_f32(bits.size, bits.ctypes.data, out.ctypes.data) != 0:
            raise ValueError("oracle rejected the arguments")
        return out

    def f16_to_f32(self, bits: np.ndarray) -> np.ndarray:
        """Widen IEEE binary16 bit patterns (uint16) to the float32 values they encode."""
        bits = np.ascontiguousarray(bits)
        if bits.dtype != np.uint16:
            raise TypeError("binary16 inputs must be uint16 bit patterns, got %s" % bits.dtype)
        out = np.empty(bits.shape, dtype=np.float32)
        if self.lib.t2s_oracle_f16_to_f32(bits.size, bits.ctypes.data, out.ctypes.data) != 0:
            raise ValueError("oracle rejected the arguments")
        return out

    def gemm_f16(self, A_bits: np.ndarray, B_bits: np.ndarray) -> np.ndarray:
        """C (float32) = A x B for binary16 A, B: the FP32 definition on the widened values."""
        return self.sgemm(self.f16_to_f32(A_bits), self.f16_to_f32(B_bits), MUL_ADD)

    def gemm_f16_at(self, A_bits, B_bits, rows, cols) -> np.ndarray:
        """Elements C[rows[s], cols[s]] of the binary16 product, one by one."""
        return self.sgemm_at(self.f16_to_f32(A_bits), self.f16_to_f32(B_bits), rows, cols,
                             MUL_ADD)

    def gemm_bf16(self, A_bits: np.ndarray, B_bits: np.ndarray) -> np.ndarray:
        """C (float32) = A x B for bfloat16 A, B: the FP32 definition on the widened values."""
        return self.sgemm(self.bf16_to_f32(A_bits), self.bf16_to_f32(B_bits), MUL_ADD)

    def gemm_bf16_at(self, A_bits, B_bits, rows, cols) -> np.ndarray:
        """Elements C[rows[s], cols[s]] of the bfloat16 product, one by one."""
        return self.sgemm_at(self.bf16_to_f32(A_bits), self.bf16_to_f32(B_bits), rows, cols,
                             MUL_ADD)

    def dgemm(self, A: np.ndarray, B: np.ndarray, mode: int = MUL_ADD) -> np.ndarray:
        """Full FP64 product C = A x B (float64, row-major)."""
        A, B = _f64(A), _f64(B)
        M, N, K = _shapes(A, B)
        C = np.empty((M, N), dtype=np.float64)
        rc = self.lib.t2s_oracle_dgemm(M, N, K, A.ctypes.data, B.ctypes.data, C.ctypes.data,
                                       mode)
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return C

    def dgemm_at(self, A: np.ndarray, B: np.ndarray, rows, cols,
                 mode: int = MUL_ADD) -> np.ndarray:
        """Elements C[rows[s], cols[s]] of the FP64 product, one by one."""
        A, B = _f64(A), _f64(B)
        M, N, K = _shapes(A, B)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        if rows.shape != cols.shape or rows.ndim != 1:
            raise ValueError("rows and cols must be 1-D and of equal length")
        out = np.empty(rows.shape[0], dtype=np.float64)
        rc = self.lib.t2s_oracle_dgemm_at(M, N, K, A.ctypes.data, B.ctypes.data,
                                          rows.shape[0], rows.ctypes.data, cols.ctypes.data,
                                          out.ctypes.data, mode)
        if rc != 0:
            raise ValueError("oracle rejected the arguments")
        return out


def _f32(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("oracle inputs must be float32, got %s" % x.dtype)
    return x


def _f64(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.float64:
        raise TypeError("FP64 oracle inputs must be float64, got %s" % x.dtype)
    return x


def _shapes(A: np.ndarray, B: np.ndarray):
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch: A %s, B %s" % (A.shape, B.shape))
    return A.shape[0], B.shape[1], A.shape[1]


def default() -> Oracle:
    """The oracle built from ``gemm_oracle.c`` as committed."""
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def sgemm(A, B, mode: int = MUL_ADD) -> np.ndarray:
    return default().sgemm(A, B, mode)


def sgemm_at(A, B, rows, cols, mode: int = MUL_ADD) -> np.ndarray:
    return default().sgemm_at(A, B, rows, cols, mode)


def sgemm_rows(A, B, r0: int, r1: int, mode: int = MUL_ADD) -> np.ndarray:
    return default().sgemm_rows(A, B, r0, r1, mode)


def vector_add(x, y) -> np.ndarray:
    return default().vector_add(x, y)


def bf16_to_f32(bits) -> np.ndarray:
    return default().bf16_to_f32(bits)


def gemm_bf16(A_bits, B_bits) -> np.ndarray:
    return default().gemm_bf16(A_bits, B_bits)


def gemm_bf16_at(A_bits, B_bits, rows, cols) -> np.ndarray:
    return default().gemm_bf16_at(A_bits, B_bits, rows, cols)


def f16_to_f32(bits) -> np.ndarray:
    return default().f16_to_f32(bits)


def gemm_f16(A_bits, B_bits) -> np.ndarray:
    return default().gemm_f16(A_bits, B_bits)


def gemm_f16_at(A_bits, B_bits, rows, cols) -> np.ndarray:
    return default().gemm_f16_at(A_bits, B_bits, rows, cols)


def dgemm(A, B, mode: int = MUL_ADD) -> np.ndarray:
    return default().dgemm(A, B, mode)


def dgemm_at(A, B, rows, cols, mode: int = MUL_ADD) -> np.ndarray:
    return default().dgemm_at(A, B, rows, cols, mode)


def num_threads() -> int:
    """Host threads the oracle uses (OpenMP)."""
    return default().lib.t2s_oracle_num_threads()


def set_num_threads(n: int) -> None:
    default().lib.t2s_oracle_set_num_threads(int(n))
