"""Maximum-size cases (GPU): outputs and vectors beyond 2^31 elements, so that every index
on the path must be 64-bit. Inputs are small in K; results are checked on sampled elements
gathered on the device (the full C of 10 GB never leaves it)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from roofline_driven_tiling_gb300 import binding, inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    assert binding.device_status() == binding.T2S_OK


def sample(M, N, seed, n=20000):
    rng = np.random.default_rng(seed)
    rows = np.concatenate([rng.integers(0, M, n), [M - 1, M - 1, 0], rng.integers(M - 130, M, 500)])
    cols = np.concatenate([rng.integers(0, N, n), [N - 1, 0, N - 1], rng.integers(0, N, 500)])
    return rows, cols


def gather(C, rows, cols):
    r = torch.from_numpy(rows).cuda()
    c = torch.from_numpy(cols).cuda()
    return C[r, c].cpu().numpy()


def test_product_c_beyond_2_31_elements():
    M, N, K = 65536, 40000, 32  # C: 2.6e9 elements (10.5 GB)
    A, B = inputs.uniform(M, K, 71), inputs.uniform(K, N, 72)
    C = binding.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    assert binding.device_status() == binding.T2S_OK
    rows, cols = sample(M, N, 1)
    want = oracle.sgemm_at(A, B, rows, cols, oracle.FMA)
    assert np.array_equal(gather(C, rows, cols).view(np.uint32), want.view(np.uint32))
    del C
    torch.cuda.empty_cache()


def test_bf16_c_beyond_2_31_elements():
    M, N, K = 65536, 40000, 64
    Ab, Bb = inputs.uniform_bf16(M, K, 73), inputs.uniform_bf16(K, N, 74)
    dA = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.bfloat16)
    dB = torch.from_numpy(Bb.view(np.int16)).cuda().view(torch.bfloat16)
    C = binding.gemm_bf16(dA, dB)
    assert binding.device_status() == binding.T2S_OK
    rows, cols = sample(M, N, 2)
    want = oracle.gemm_bf16_at(Ab, Bb, rows, cols)
    A32, B32 = oracle.bf16_to_f32(Ab), oracle.bf16_to_f32(Bb)
    tol = 1e-6 * K * float(np.abs(A32).max()) * float(np.abs(B32).max())
    assert float(np.max(np.abs(gather(C, rows, cols) - want))) <= tol
    del C
    torch.cuda.empty_cache()


def test_streamk_c_beyond_2_31_elements():
    M, N, K = 65536, 36000, 64
    A, B = inputs.uniform(M, K, 75), inputs.uniform(K, N, 76)
    C = binding.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), kernel="streamk")
    assert binding.device_status() == binding.T2S_OK
    rows, cols = sample(M, N, 3)
    want = oracle.sgemm_at(A, B, rows, cols, oracle.FMA)
    tol = 1e-6 * K * float(np.abs(A).max()) * float(np.abs(B).max())
    assert float(np.max(np.abs(gather(C, rows, cols) - want))) <= tol
    del C
    torch.cuda.empty_cache()


def test_vector_add_beyond_2_31_elements():
    n = (1 << 31) + 37
    x = torch.empty(n, dtype=torch.float32, device="cuda").uniform_(-1, 1)
    y = torch.empty(n, dtype=torch.float32, device="cuda").uniform_(-1, 1)
    z = torch.empty(n, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert binding.t2s_vector_add_f32(n, x.data_ptr(), y.data_ptr(), z.data_ptr(), s) == binding.T2S_OK
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    idx = torch.from_numpy(np.concatenate([rng.integers(0, n, 100000), np.arange(n - 64, n)])).cuda()
    xs, ys, zs = x[idx].cpu().numpy(), y[idx].cpu().numpy(), z[idx].cpu().numpy()
    assert np.array_equal(zs.view(np.uint32), oracle.vector_add(xs, ys).view(np.uint32))
