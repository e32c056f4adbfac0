"""GB300-native (sm_103a) FP32 matrix multiply C = A x B, row-major.

The compute path is the CUDA library ``libt2s_gemm.so`` (C ABI in
``include/t2s_gemm.h``); ``binding`` is its ctypes binding. ``roofline`` holds the
performance model used for reporting and ``inputs`` the seeded synthetic inputs.
"""
from . import binding, inputs, roofline  # noqa: F401
from .binding import gemm, gemm_bf16, gemm_f16, gemm_f64, device_status, plan  # noqa: F401

__all__ = ["binding", "inputs", "roofline", "gemm", "gemm_bf16", "gemm_f16", "gemm_f64",
           "device_status", "plan"]
