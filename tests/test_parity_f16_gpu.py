"""Parity of the FP16 tensor-core product (t2s_gemm_f16_f32) with the oracle (GPU tests).

The same bars as for BF16: products of two binary16 values are exact in FP32, so wherever
every partial sum is exact (the integer pattern, dyadic values, subnormal operands scaled by
integers) C must equal the oracle's FP32 definition on the widened inputs bit for bit;
otherwise max |C - C_oracle| <= 1e-6 * K * max|a| * max|b|.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import test_parity_bf16_gpu as h
from roofline_driven_tiling_gb300 import binding, inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F16_NAN = 0x7E00


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    assert binding.device_status() == binding.T2S_OK


def run_f16(Ab: np.ndarray, Bb: np.ndarray, shift: int = 0) -> np.ndarray:
    """The product through the C ABI on guarded device buffers (canaries around A and B,
    sentinels around C)."""
    M, K = Ab.shape
    N = Bb.shape[1]
    dA, dB = h.GuardedBits(Ab, shift), h.GuardedBits(Bb, shift)
    c = torch.full((M * N + 2 * h.GUARD,), float(h.C_SENTINEL), dtype=torch.float32,
                   device="cuda")
    need = binding.t2s_gemm_f16_f32_workspace_size(M, N, K)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = binding.t2s_gemm_f16_f32(M, N, K, dA.ptr, dB.ptr, c.data_ptr() + 4 * h.GUARD,
                                  ws.data_ptr(), ws.numel(), s)
    assert rc == binding.T2S_OK, binding.status_string(rc)
    assert binding.t2s_device_status(s) == binding.T2S_OK
    host = c.cpu().numpy()
    assert dA.intact() and dB.intact()
    assert np.all(host[:h.GUARD] == h.C_SENTINEL) and np.all(host[h.GUARD + M * N:] == h.C_SENTINEL)
    return host[h.GUARD:h.GUARD + M * N].reshape(M, N)


def tolerance(Ab, Bb) -> float:
    A, B = oracle.f16_to_f32(Ab), oracle.f16_to_f32(Bb)
    return 1e-6 * Ab.shape[1] * float(np.max(np.abs(A))) * float(np.max(np.abs(B)))


@pytest.mark.parametrize("shape", [(256, 256, 256), (1000, 1003, 997), (389, 512, 256),
                                   (129, 64, 24)], ids=lambda s: "x".join(map(str, s)))
def test_f16_integer_pattern_exact(shape):
    M, N, K = shape
    A, B = inputs.integer_pattern(M, N, K)
    Ab, Bb = inputs.to_f16_bits(A), inputs.to_f16_bits(B)
    assert h.bits_equal(run_f16(Ab, Bb), oracle.gemm_f16(Ab, Bb))


def test_f16_partial_last_round_exact():
    """The BF16 partial-round case for binary16: 80 pair tiles on 76 pairs, integer operands."""
    M, N, K = 2560, 2048, 4096
    A, B = inputs.integer_pattern(M, N, K)
    Ab, Bb = inputs.to_f16_bits(A), inputs.to_f16_bits(B)
    dA = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.float16)
    dB = torch.from_numpy(Bb.view(np.int16)).cuda().view(torch.float16)
    C = binding.gemm_f16(dA, dB)
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = h.split_round_positions(M, N, np.random.default_rng(6))
    assert h.bits_equal(C[rows, cols], oracle.gemm_f16_at(Ab, Bb, rows, cols))


@pytest.mark.parametrize("kind", ["integer", "uniform"])
def test_f16_wide_tiles_ragged_edges(kind):
    """The BF16 ragged wide-tile case for binary16: 2500 x 2000 x 3000 on 256 x 512 pair
    tiles, partial tiles at the bottom and right edges and a partial last k block."""
    M, N, K = 2500, 2000, 3000
    if kind == "integer":
        A, B = inputs.integer_pattern(M, N, K)
        Ab, Bb = inputs.to_f16_bits(A), inputs.to_f16_bits(B)
    else:
        Ab, Bb = inputs.uniform_f16(M, K, 1008), inputs.uniform_f16(K, N, 2008)
    dA = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.float16)
    dB = torch.from_numpy(Bb.view(np.int16)).cuda().view(torch.float16)
    C = binding.gemm_f16(dA, dB)
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = h.edge_positions(M, N, np.random.default_rng(10))
    ref = oracle.gemm_f16_at(Ab, Bb, rows, cols)
    if kind == "integer":
        assert h.bits_equal(C[rows, cols], ref)
    else:
        assert float(np.max(np.abs(C[rows, cols] - ref))) <= tolerance(Ab, Bb)


def test_f16_dyadic_exact_misaligned():
    A = inputs.dyadic(300, 77, seed=31, denom=256, span=1000)
    B = inputs.dyadic(77, 192, seed=32, denom=16, span=64)
    Ab, Bb = inputs.to_f16_bits(A), inputs.to_f16_bits(B)
    for shift in (0, 1, 3):
        assert h.bits_equal(run_f16(Ab, Bb, shift), oracle.gemm_f16(Ab, Bb))


def test_f16_subnormal_operands_exact():
    """Subnormal binary16 operands (multiples of 2^-24) times small integers: every product
    and sum is exact in FP32, so a tensor core that flushed subnormals would be caught."""
    M, N, K = 260, 136, 96
    rng = np.random.default_rng(3)
    a_bits = rng.integers(1, 0x400, size=(M, K)).astype(np.uint16)  # all subnormal
    a_bits[rng.random((M, K)) < 0.5] |= np.uint16(0x8000)
    B = inputs.integer_pattern(1, N, K)[1]
    Bb = inputs.to_f16_bits(B)
    assert h.bits_equal(run_f16(a_bits, Bb), oracle.gemm_f16(a_bits, Bb))


def test_f16_ragged_tolerance():
    M, N, K = 1000, 1003, 997
    Ab, Bb = inputs.uniform_f16(M, K, 1013), inputs.uniform_f16(K, N, 2013)
    C = run_f16(Ab, Bb)
    assert float(np.max(np.abs(C - oracle.gemm_f16(Ab, Bb)))) <= tolerance(Ab, Bb)


@pytest.mark.parametrize("shift", [0, 1], ids=["aligned", "misaligned"])
@pytest.mark.parametrize("shape", h.small_shapes()[::2], ids=lambda s: "x".join(map(str, s)))
def test_f16_small_shapes(shape, shift):
    M, N, K = shape
    Ab, Bb = inputs.uniform_f16(M, K, 41 + M), inputs.uniform_f16(K, N, 43 + N)
    C = run_f16(Ab, Bb, shift)
    assert float(np.max(np.abs(C - oracle.gemm_f16(Ab, Bb)))) <= tolerance(Ab, Bb)


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (8192, 8192, 8192), (16384, 16384, 32),
                                   (256, 256, 65536), (1280, 1024, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_f16_large_sampled(shape):
    M, N, K = shape
    Ab, Bb = inputs.uniform_f16(M, K, 1006), inputs.uniform_f16(K, N, 2006)
    dA = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.float16)
    dB = torch.from_numpy(Bb.view(np.int16)).cuda().view(torch.float16)
    C = binding.gemm_f16(dA, dB)
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = h.sample_positions(M, N, np.random.default_rng(M + 3 * K))
    ref = oracle.gemm_f16_at(Ab, Bb, rows, cols)
    assert float(np.max(np.abs(C[rows, cols] - ref))) <= tolerance(Ab, Bb)


def test_f16_nan_and_inf_propagate():
    M, N, K = 130, 144, 96
    A = inputs.dyadic(M, K, seed=51, denom=4, span=8)
    B = np.abs(inputs.dyadic(K, N, seed=52, denom=4, span=8)) + np.float32(0.25)
    Ab, Bb = inputs.to_f16_bits(A), inputs.to_f16_bits(B)
    Ab[5, 17] = F16_NAN
    Ab[77, 90] = 0x7C00  # +inf; every B entry is positive, so row 77 is +inf
    C = run_f16(Ab, Bb)
    assert np.all(np.isnan(C[5])) and np.all(np.isposinf(C[77]))
    rest = np.ones(M, bool)
    rest[[5, 77]] = False
    assert h.bits_equal(C[rest], oracle.gemm_f16(Ab, Bb)[rest])
