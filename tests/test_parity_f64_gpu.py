"""Parity of the FP64 kernels (t2s_gemm_f64, _naive, _smem32) with the FP64 oracle (GPU tests).

Every FP64 kernel sums each element with one fused multiply-add per k in ascending k, so it
must equal the oracle's FMA reading bit for bit on every input (NaN payloads aside: NaN
positions must agree); on the integer pattern, where every step is exact, it must also equal
the two-rounding reading.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from roofline_driven_tiling_gb300 import binding, inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KERNELS = ("ffma", "naive", "smem32")
GUARD = 32
SENTINEL = -12345.678


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    assert binding.device_status() == binding.T2S_OK


def guarded(x: np.ndarray, fill: float):
    buf = torch.full((x.size + 2 * GUARD,), fill, dtype=torch.float64, device="cuda")
    if x.size:
        buf[GUARD:GUARD + x.size] = torch.from_numpy(np.ascontiguousarray(x).ravel()).cuda()
    return buf


def run(kernel: str, A: np.ndarray, B: np.ndarray, stream=None) -> np.ndarray:
    M, K = A.shape
    N = B.shape[1]
    dA, dB = guarded(A, float("nan")), guarded(B, float("nan"))
    dC = guarded(np.full((M, N), SENTINEL), SENTINEL)
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    fn = getattr(binding, binding.KERNELS_F64[kernel])
    rc = fn(M, N, K, dA.data_ptr() + 8 * GUARD, dB.data_ptr() + 8 * GUARD,
            dC.data_ptr() + 8 * GUARD, s)
    assert rc == binding.T2S_OK, binding.status_string(rc)
    assert binding.t2s_device_status(s) == binding.T2S_OK
    host = dC.cpu().numpy()
    assert np.all(host[:GUARD] == SENTINEL) and np.all(host[GUARD + M * N:] == SENTINEL), \
        "write outside C"
    return host[GUARD:GUARD + M * N].reshape(M, N)


def same_bits(x: np.ndarray, y: np.ndarray) -> bool:
    nx, ny = np.isnan(x), np.isnan(y)
    return bool(np.array_equal(nx, ny) and
                np.array_equal(x[~nx].view(np.uint64), y[~ny].view(np.uint64)))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("n", [256, 1024])
def test_f64_integer_pattern_exact(kernel, n):
    A, B = inputs.integer_pattern(n, n, n)
    A, B = A.astype(np.float64), B.astype(np.float64)
    C = run(kernel, A, B)
    for mode in (oracle.FMA, oracle.MUL_ADD):
        assert same_bits(C, oracle.dgemm(A, B, mode))


@pytest.mark.parametrize("kernel", KERNELS)
def test_f64_ragged_uniform_bit_exact(kernel):
    M, N, K = 300, 301, 297
    A, B = inputs.uniform_f64(M, K, 3001), inputs.uniform_f64(K, N, 3002)
    assert same_bits(run(kernel, A, B), oracle.dgemm(A, B, oracle.FMA))


def small_shapes():
    edge = [1, 2, 3, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129]
    rng = np.random.default_rng(77)
    shapes = {(1, 1, 1), (1, 1, 129), (129, 1, 1), (1, 129, 1), (64, 64, 16), (65, 65, 17)}
    while len(shapes) < 40:
        shapes.add(tuple(int(x) for x in rng.choice(edge, 3)))
    return sorted(shapes)


@pytest.mark.parametrize("shape", small_shapes(), ids=lambda s: "x".join(map(str, s)))
def test_f64_small_shapes(shape):
    M, N, K = shape
    A, B = inputs.uniform_f64(M, K, 11 + M), inputs.uniform_f64(K, N, 13 + N)
    want = oracle.dgemm(A, B, oracle.FMA)
    for kernel in KERNELS:
        assert same_bits(run(kernel, A, B), want), kernel


def test_f64_special_values():
    M, N, K = 70, 90, 40
    rng = np.random.default_rng(5)
    A = inputs.uniform_f64(M, K, 41) * 1e300
    B = inputs.uniform_f64(K, N, 42)
    specials = np.array([np.inf, -np.inf, np.nan, -0.0, 5e-324, -2.5e-308, 1e308])
    for X in (A, B):
        pos = rng.integers(0, X.size, 60)
        X.ravel()[pos] = specials[rng.integers(0, specials.size, 60)]
    want = oracle.dgemm(A, B, oracle.FMA)
    for kernel in KERNELS:
        assert same_bits(run(kernel, A, B), want), kernel


def test_f64_large_sampled():
    M, N, K = 2048, 2048, 2048
    A, B = inputs.uniform_f64(M, K, 4001), inputs.uniform_f64(K, N, 4002)
    C = binding.gemm_f64(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()).cpu().numpy()
    assert binding.device_status() == binding.T2S_OK
    rng = np.random.default_rng(9)
    rows = np.concatenate([rng.integers(0, M, 3000), np.arange(M), np.full(N, M - 1)])
    cols = np.concatenate([rng.integers(0, N, 3000), np.full(M, N - 1), np.arange(N)])
    want = oracle.dgemm_at(A, B, rows, cols, oracle.FMA)
    assert np.array_equal(C[rows, cols].view(np.uint64), want.view(np.uint64))


def test_f64_k_zero_and_stream():
    dA = torch.zeros((0,), dtype=torch.float64, device="cuda")
    dC = torch.full((12,), 3.0, dtype=torch.float64, device="cuda")
    for kernel in KERNELS:
        fn = getattr(binding, binding.KERNELS_F64[kernel])
        assert fn(3, 4, 0, 0, 0, dC.data_ptr(), 0) == binding.T2S_OK
        torch.cuda.synchronize()
        assert torch.all(dC == 0) and not torch.any(torch.signbit(dC))
        dC.fill_(3.0)
    del dA
    s = torch.cuda.Stream()
    A, B = inputs.uniform_f64(130, 70, 51), inputs.uniform_f64(70, 66, 52)
    assert same_bits(run("ffma", A, B, stream=s), oracle.dgemm(A, B, oracle.FMA))
