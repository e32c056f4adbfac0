"""Cache-blocked multi-core CPU GEMM: the stronger CPU baseline (ctypes loader).

A BASELINE, not a checker: ``bench.py`` times it beside the plain oracle so that the GPU's
lead over a CPU is not measured against a strawman alone. No test and no product code
compares a result against it; the tests pin it, in turn, to the oracle.

The arithmetic lives in ``blocked_gemm.c`` (plain C, OpenMP); this module compiles it with
gcc and marshals numpy arrays into it. It shares no code with the oracle or the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "blocked_gemm.c")
_LIB = os.path.join(_HERE, "libcpu_blocked_gemm.so")
_CFLAGS = ["-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``blocked_gemm.c`` into ``libcpu_blocked_gemm.so`` (gcc). Returns the path."""
    with _lock:
        stale = not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + ".tmp%d" % os.getpid()
            subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        path = build()
        with _lock:
            if _lib is None:
                l = ctypes.CDLL(path)
                i64, fp = ctypes.c_int64, ctypes.c_void_p
                l.t2s_cpu_blocked_sgemm.argtypes = [i64, i64, i64, fp, fp, fp]
                l.t2s_cpu_blocked_sgemm.restype = ctypes.c_int
                l.t2s_cpu_blocked_num_threads.argtypes = []
                l.t2s_cpu_blocked_num_threads.restype = ctypes.c_int
                l.t2s_cpu_blocked_set_num_threads.argtypes = [ctypes.c_int]
                l.t2s_cpu_blocked_set_num_threads.restype = None
                _lib = l
    return _lib


def num_threads() -> int:
    return int(lib().t2s_cpu_blocked_num_threads())


def set_num_threads(n: int) -> None:
    lib().t2s_cpu_blocked_set_num_threads(int(n))


def sgemm(A: np.ndarray, B: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """C = A x B for row-major float32 A (M x K) and B (K x N) on every OpenMP thread."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch: %s x %s" % (A.shape, B.shape))
    M, K = A.shape
    N = B.shape[1]
    C = np.empty((M, N), dtype=np.float32) if out is None else out
    if C.shape != (M, N) or C.dtype != np.float32 or not C.flags.c_contiguous:
        raise ValueError("out must be a contiguous float32 array of shape (%d, %d)" % (M, N))
    rc = lib().t2s_cpu_blocked_sgemm(M, N, K, A.ctypes.data, B.ctypes.data, C.ctypes.data)
    if rc != 0:
        raise RuntimeError("t2s_cpu_blocked_sgemm failed (%d)" % rc)
    return C
