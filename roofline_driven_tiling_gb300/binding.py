"""ctypes binding of libt2s_gemm.so: the C ABI of include/t2s_gemm.h under the same names.

Argument marshalling only. Every step of the multiply runs in the CUDA library;
there is no fallback of any kind. If the library is missing the import of a
function raises, naming the build step.

The ``gemm`` helper takes torch CUDA tensors (row-major, contiguous, float32),
passes their device pointers and the current torch stream, and raises on any
non-zero status. ``t2s_*`` functions take raw integers (pointers as ints, the
stream as the integer value of a cudaStream_t).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libt2s_gemm.so")

T2S_OK = 0
T2S_ERR_INVALID = 1
T2S_ERR_CUDA = 2
T2S_ERR_TIMEOUT = 3
T2S_ERR_WORKSPACE = 4
T2S_ERR_TOO_LARGE = 5
T2S_TF32X3_NOALLOC_MAX_SCRATCH = 32 << 20
T2S_MAX_DIM = 1 << 30

#: Every function the header declares, with (argtypes, restype).
_i64, _p, _i, _sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "t2s_gemm_f32": ([_i64, _i64, _i64, _p, _p, _p, _p], _i),
    "t2s_gemm_f32_host": ([_i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p], _i),
    "t2s_gemm_f32_plan": ([_i64, _i64, _i64, _i], _i),
    "t2s_gemm_f32_splitk_plan": ([_i64, _i64, _i64, _i], _i),
    "t2s_gemm_f32_naive": ([_i64, _i64, _i64, _p, _p, _p, _p], _i),
    "t2s_gemm_f32_smem32": ([_i64, _i64, _i64, _p, _p, _p, _p], _i),
    "t2s_gemm_f32_splitk_workspace_size": ([_i64, _i64, _i64, _i], _sz),
    "t2s_gemm_f32_splitk": ([_i64, _i64, _i64, _p, _p, _p, _i, _p, _sz, _p], _i),
    "t2s_gemm_f32_streamk_workspace_size": ([_i64, _i64, _i64], _sz),
    "t2s_gemm_f32_streamk": ([_i64, _i64, _i64, _p, _p, _p, _p, _sz, _p], _i),
    "t2s_gemm_f32_tf32x3_workspace_size": ([_i64, _i64, _i64], _sz),
    "t2s_gemm_f32_tf32x3": ([_i64, _i64, _i64, _p, _p, _p, _p, _sz, _p], _i),
    "t2s_gemm_f32_tf32x3_noalloc": ([_i64, _i64, _i64, _p, _p, _p, _p], _i),
    "t2s_gemm_f64": ([_i64, _i64, _i64, _p, _p, _p, _p], _i),
    "t2s_gemm_f64_naive": ([_i64, _i64, _i64, _p, _p, _p, _p], _i),
    "t2s_gemm_f64_smem32": ([_i64, _i64, _i64, _p, _p, _p, _p], _i),
    "t2s_gemm_bf16_f32_workspace_size": ([_i64, _i64, _i64], _sz),
    "t2s_gemm_bf16_f32": ([_i64, _i64, _i64, _p, _p, _p, _p, _sz, _p], _i),
    "t2s_gemm_f16_f32_workspace_size": ([_i64, _i64, _i64], _sz),
    "t2s_gemm_f16_f32": ([_i64, _i64, _i64, _p, _p, _p, _p, _sz, _p], _i),
    "t2s_vector_add_f32": ([_i64, _p, _p, _p, _p], _i),
    "t2s_status_string": ([_i], ctypes.c_char_p),
    "t2s_device_status": ([_p], _i),
    "t2s_last_cuda_error": ([], _i),
    "t2s_selftest_wait_timeout": ([_i64, _p], _i),
    "t2s_probe_outputs": ([], _i),
    "t2s_probe_fp32_fma": ([_i64, _p, _p, _p], _i),
    "t2s_probe_tf32_mma": ([_i64, _p, _p, _p], _i),
    "t2s_probe_store_f32": ([_i64, _i64, _p, _i, ctypes.c_float, _p, _p], _i),
    "t2s_version": ([], _i),
}

_lib = None


class T2SError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = "%s failed: %s" % (what, status_string(status))
        if status == T2S_ERR_CUDA:
            msg += " (cudaError %d)" % lib().t2s_last_cuda_error()
        super().__init__(msg)


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libt2s_gemm.so is not built: run "
                              "`python -c 'import __graft_entry__ as g; g.build()'` first")
        l = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = res
        _lib = l
    return _lib


# ---- the C ABI, same names ------------------------------------------------------------
def t2s_gemm_f32(M, N, K, A, B, C, stream=0) -> int:
    return lib().t2s_gemm_f32(M, N, K, A, B, C, stream)


def t2s_gemm_f32_host(M, N, K, hA, hB, hC, dA, dB, dC, stream=0) -> int:
    return lib().t2s_gemm_f32_host(M, N, K, hA, hB, hC, dA, dB, dC, stream)


def t2s_gemm_f32_plan(M, N, K, sms) -> int:
    return lib().t2s_gemm_f32_plan(M, N, K, sms)


def t2s_gemm_f32_splitk_plan(M, N, K, sms) -> int:
    return lib().t2s_gemm_f32_splitk_plan(M, N, K, sms)


def t2s_gemm_f32_naive(M, N, K, A, B, C, stream=0) -> int:
    return lib().t2s_gemm_f32_naive(M, N, K, A, B, C, stream)


def t2s_gemm_f32_smem32(M, N, K, A, B, C, stream=0) -> int:
    return lib().t2s_gemm_f32_smem32(M, N, K, A, B, C, stream)


def t2s_gemm_f32_splitk_workspace_size(M, N, K, splits=0) -> int:
    return lib().t2s_gemm_f32_splitk_workspace_size(M, N, K, splits)


def t2s_gemm_f32_splitk(M, N, K, A, B, C, splits, workspace, workspace_bytes, stream=0) -> int:
    return lib().t2s_gemm_f32_splitk(M, N, K, A, B, C, splits, workspace, workspace_bytes, stream)


def t2s_gemm_f32_streamk_workspace_size(M, N, K) -> int:
    return lib().t2s_gemm_f32_streamk_workspace_size(M, N, K)


def t2s_gemm_f32_streamk(M, N, K, A, B, C, workspace, workspace_bytes, stream=0) -> int:
    return lib().t2s_gemm_f32_streamk(M, N, K, A, B, C, workspace, workspace_bytes, stream)


def t2s_gemm_f32_tf32x3_workspace_size(M, N, K) -> int:
    return lib().t2s_gemm_f32_tf32x3_workspace_size(M, N, K)


def t2s_gemm_f32_tf32x3(M, N, K, A, B, C, workspace, workspace_bytes, stream=0) -> int:
    return lib().t2s_gemm_f32_tf32x3(M, N, K, A, B, C, workspace, workspace_bytes, stream)


def t2s_gemm_f32_tf32x3_noalloc(M, N, K, A, B, C, stream=0) -> int:
    """3xTF32 product with the library's built-in scratch array (no allocation)."""
    return lib().t2s_gemm_f32_tf32x3_noalloc(M, N, K, A, B, C, stream)


def t2s_gemm_f64(M, N, K, A, B, C, stream=0) -> int:
    return lib().t2s_gemm_f64(M, N, K, A, B, C, stream)


def t2s_gemm_f64_naive(M, N, K, A, B, C, stream=0) -> int:
    return lib().t2s_gemm_f64_naive(M, N, K, A, B, C, stream)


def t2s_gemm_f64_smem32(M, N, K, A, B, C, stream=0) -> int:
    return lib().t2s_gemm_f64_smem32(M, N, K, A, B, C, stream)


def t2s_gemm_bf16_f32_workspace_size(M, N, K) -> int:
    return lib().t2s_gemm_bf16_f32_workspace_size(M, N, K)


def t2s_gemm_bf16_f32(M, N, K, A, B, C, workspace, workspace_bytes, stream=0) -> int:
    return lib().t2s_gemm_bf16_f32(M, N, K, A, B, C, workspace, workspace_bytes, stream)


def t2s_gemm_f16_f32_workspace_size(M, N, K) -> int:
    return lib().t2s_gemm_f16_f32_workspace_size(M, N, K)


def t2s_gemm_f16_f32(M, N, K, A, B, C, workspace, workspace_bytes, stream=0) -> int:
    return lib().t2s_gemm_f16_f32(M, N, K, A, B, C, workspace, workspace_bytes, stream)


def t2s_vector_add_f32(n, x, y, z, stream=0) -> int:
    return lib().t2s_vector_add_f32(n, x, y, z, stream)


def t2s_status_string(status: int) -> str:
    return lib().t2s_status_string(status).decode()


def t2s_device_status(stream=0) -> int:
    return lib().t2s_device_status(stream)


def t2s_last_cuda_error() -> int:
    return lib().t2s_last_cuda_error()


def t2s_selftest_wait_timeout(limit_ns: int, stream=0) -> int:
    return lib().t2s_selftest_wait_timeout(limit_ns, stream)


def t2s_version() -> int:
    return lib().t2s_version()


def t2s_probe_outputs() -> int:
    return lib().t2s_probe_outputs()


def probe(kind: str, iters: int, out_ptr: int, stream=0) -> int:
    """Launches a throughput probe ("fp32_fma" or "tf32_mma") on `stream`; returns the FLOPs
    of the launch (raises T2SError on a bad status)."""
    flops = ctypes.c_int64(0)
    fn = lib().t2s_probe_fp32_fma if kind == "fp32_fma" else lib().t2s_probe_tf32_mma
    rc = fn(iters, out_ptr, ctypes.addressof(flops), stream)
    if rc != T2S_OK:
        raise T2SError(rc, "t2s_probe_" + kind)
    return int(flops.value)


def probe_store(M: int, N: int, c_ptr: int, mode: int, value: float = 0.0, stream=0) -> int:
    """Launches the store-path probe on `stream`: writes `value` to the M x N matrix at c_ptr
    in the short-K product's store pattern (mode 0: TMA boxes, 1: 16-byte stores from
    registers); returns the bytes written (raises T2SError on a bad status)."""
    nbytes = ctypes.c_int64(0)
    rc = lib().t2s_probe_store_f32(M, N, c_ptr, mode, value, ctypes.addressof(nbytes), stream)
    if rc != T2S_OK:
        raise T2SError(rc, "t2s_probe_store_f32")
    return int(nbytes.value)


status_string = t2s_status_string

# ---- torch convenience ----------------------------------------------------------------
KERNELS = {
    "ffma": "t2s_gemm_f32",
    "naive": "t2s_gemm_f32_naive",
    "smem32": "t2s_gemm_f32_smem32",
    "tf32x3": "t2s_gemm_f32_tf32x3",
    "streamk": "t2s_gemm_f32_streamk",
}


def _check(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError("%s must be a float32 CUDA tensor" % name)
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous 2-D (row-major) tensor" % name)


def gemm(A, B, out=None, kernel: str = "ffma", workspace=None, stream=None):
    """C = A @ B through the library (torch tensors in, torch tensor out).

    `kernel` is one of "ffma" (the product), "naive", "smem32", "tf32x3", "streamk". For
    "tf32x3" and "streamk" a workspace tensor is allocated here (by torch) unless one is passed.
    """
    import torch
    _check(A, "A")
    _check(B, "B")
    if A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(out, "out")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be %d x %d" % (M, N))
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    fn = getattr(lib(), KERNELS[kernel])
    if kernel in ("tf32x3", "streamk"):
        need = getattr(lib(), KERNELS[kernel] + "_workspace_size")(M, N, K)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=A.device)
        rc = fn(M, N, K, A.data_ptr(), B.data_ptr(), out.data_ptr(), workspace.data_ptr(),
                workspace.numel() * workspace.element_size(), stream)
    else:
        rc = fn(M, N, K, A.data_ptr(), B.data_ptr(), out.data_ptr(), stream)
    if rc != T2S_OK:
        raise T2SError(rc, KERNELS[kernel])
    return out


KERNELS_F64 = {
    "ffma": "t2s_gemm_f64",
    "naive": "t2s_gemm_f64_naive",
    "smem32": "t2s_gemm_f64_smem32",
}


def gemm_f64(A, B, out=None, kernel: str = "ffma", stream=None):
    """C = A @ B for float64 CUDA tensors (row-major); `kernel` as for ``gemm``."""
    import torch
    for t, name in ((A, "A"), (B, "B")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float64:
            raise TypeError("%s must be a float64 CUDA tensor" % name)
        if t.dim() != 2 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous 2-D (row-major) tensor" % name)
    if A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float64, device=A.device)
    if (not isinstance(out, torch.Tensor) or out.dtype != torch.float64 or not out.is_cuda
            or not out.is_contiguous() or tuple(out.shape) != (M, N)):
        raise ValueError("out must be a contiguous float64 CUDA tensor of %d x %d" % (M, N))
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    name = KERNELS_F64[kernel]
    rc = getattr(lib(), name)(M, N, K, A.data_ptr(), B.data_ptr(), out.data_ptr(), stream)
    if rc != T2S_OK:
        raise T2SError(rc, name)
    return out


def _gemm_16bit(A, B, out, workspace, stream, dtype, name):
    import torch
    for t, what in ((A, "A"), (B, "B")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype:
            raise TypeError("%s must be a %s CUDA tensor" % (what, dtype))
        if t.dim() != 2 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous 2-D (row-major) tensor" % what)
    if A.shape[1] != B.shape[0]:
        raise ValueError("shape mismatch: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(out, "out")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be %d x %d" % (M, N))
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    l = lib()
    need = getattr(l, name + "_workspace_size")(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=A.device)
    rc = getattr(l, name)(M, N, K, A.data_ptr(), B.data_ptr(), out.data_ptr(),
                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          stream)
    if rc != T2S_OK:
        raise T2SError(rc, name)
    return out


def gemm_bf16(A, B, out=None, workspace=None, stream=None):
    """C (float32) = A @ B for bfloat16 CUDA tensors A (M x K) and B (K x N), row-major."""
    import torch
    return _gemm_16bit(A, B, out, workspace, stream, torch.bfloat16, "t2s_gemm_bf16_f32")


def gemm_f16(A, B, out=None, workspace=None, stream=None):
    """C (float32) = A @ B for float16 CUDA tensors A (M x K) and B (K x N), row-major."""
    import torch
    return _gemm_16bit(A, B, out, workspace, stream, torch.float16, "t2s_gemm_f16_f32")


def plan(M: int, N: int, K: int, sms: int = None) -> str:
    """The CTA tiling ``gemm`` takes for an M x N x K product, by name (host-only; `sms`
    defaults to the current device's multiprocessor count)."""
    if sms is None:
        import torch
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    code = lib().t2s_gemm_f32_plan(M, N, K, sms)
    if code < 0:
        raise ValueError("invalid shape or SM count")
    return PLAN_NAMES[code]


PLAN_NAMES = {
    0: "128x128 tiles, unrolled k loop",
    1: "128x128 tiles, compact k loop",
    2: "128x64 tiles",
    3: "64x64 tiles",
    4: "256x128 tiles",
    5: "256x128 tiles in whole rounds, the rest as 64x64 tiles",
    6: "128x128 tiles of 8 warps",
    7: "128x64 tiles of 8 warps",
    8: "128x128 tiles on a persistent grid",
    9: "56x128 tiles of 8 warps",
    10: "32x32 tiles",
    11: "256x128 tiles on a persistent grid with TMA stores of C",
}


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    return t2s_device_status(stream)
