"""Parity of the BF16 tensor-core product (t2s_gemm_bf16_f32) with the oracle (GPU tests).

Bars: products of two bfloat16 values are exact in FP32, so wherever every partial sum is
exact too (the integer pattern, small dyadic values) C must equal the oracle's FP32
definition on the widened inputs bit for bit; otherwise the tensor core's summation order
differs from ascending k and the bound is max |C - C_oracle| <= 1e-6 * K * max|a| * max|b|.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from roofline_driven_tiling_gb300 import binding, inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 64
BF16_NAN = 0x7FC0
C_SENTINEL = np.float32(-12345.678)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    assert binding.device_status() == binding.T2S_OK


class GuardedBits:
    """Device copy of a uint16 matrix between NaN canaries; `shift` extra elements of offset
    leave the data 2-byte aligned only."""

    def __init__(self, bits: np.ndarray, shift: int = 0):
        self.shape, self.n, self.start = bits.shape, bits.size, GUARD + shift
        host = np.full(self.n + 2 * GUARD + shift, BF16_NAN, dtype=np.uint16)
        host[self.start:self.start + self.n] = bits.ravel()
        self.buf = torch.from_numpy(host.view(np.int16)).cuda()

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + 2 * self.start

    def intact(self) -> bool:
        host = self.buf.cpu().numpy().view(np.uint16)
        return bool(np.all(host[:self.start] == BF16_NAN) and
                    np.all(host[self.start + self.n:] == BF16_NAN))


def run_bf16(Ab: np.ndarray, Bb: np.ndarray, shift: int = 0) -> np.ndarray:
    M, K = Ab.shape
    N = Bb.shape[1]
    dA, dB = GuardedBits(Ab, shift), GuardedBits(Bb, shift)
    c = torch.full((M * N + 2 * GUARD,), float(C_SENTINEL), dtype=torch.float32, device="cuda")
    need = binding.t2s_gemm_bf16_f32_workspace_size(M, N, K)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = binding.t2s_gemm_bf16_f32(M, N, K, dA.ptr, dB.ptr, c.data_ptr() + 4 * GUARD,
                                   ws.data_ptr(), ws.numel(), s)
    assert rc == binding.T2S_OK, binding.status_string(rc)
    assert binding.t2s_device_status(s) == binding.T2S_OK
    host = c.cpu().numpy()
    assert dA.intact() and dB.intact()
    assert np.all(host[:GUARD] == C_SENTINEL) and np.all(host[GUARD + M * N:] == C_SENTINEL), \
        "write outside C"
    return host[GUARD:GUARD + M * N].reshape(M, N)


def tolerance(Ab, Bb) -> float:
    A, B = oracle.bf16_to_f32(Ab), oracle.bf16_to_f32(Bb)
    return 1e-6 * Ab.shape[1] * float(np.max(np.abs(A))) * float(np.max(np.abs(B)))


def bits_equal(x, y) -> bool:
    return np.array_equal(x.view(np.uint32), y.view(np.uint32))


def bf16_tensor(bits: np.ndarray):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def sample_positions(M, N, rng, n_random=4096):
    rows = [0, M - 1, M // 2]
    cols = [0, N - 1, N // 2]
    r = [np.full(N, i) for i in rows] + [np.arange(M) for _ in cols]
    c = [np.arange(N) for _ in rows] + [np.full(M, j) for j in cols]
    r.append(rng.integers(0, M, n_random))
    c.append(rng.integers(0, N, n_random))
    return np.concatenate(r), np.concatenate(c)


def split_round_positions(M, N, rng):
    """The bottom-right 512 x 512 corner (the tiles of the last, partial round of the
    persistent grid when 256 x 256 pair tiles do not fill whole rounds, as in 2560 x 2048 on
    76 SM pairs), the last row and column, and random positions."""
    r0, c0 = M - 512, N - 512
    rr, cc = np.meshgrid(np.arange(r0, M), np.arange(c0, N), indexing="ij")
    rows = [rr.ravel(), np.full(N, M - 1), np.arange(M), rng.integers(0, M, 4096)]
    cols = [cc.ravel(), np.arange(N), np.full(M, N - 1), rng.integers(0, N, 4096)]
    return np.concatenate(rows), np.concatenate(cols)


def test_bf16_partial_last_round_exact():
    """2560 x 2048 x 4096: 80 pair tiles on 76 pairs, so 4 clusters run a second tile, two K
    chunks each. Integer-valued operands make every sum exact: those tiles must equal the
    definition bit for bit, like the others."""
    M, N, K = 2560, 2048, 4096
    A, B = inputs.integer_pattern(M, N, K)
    Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    dA = torch.from_numpy(Ab.view(np.int16)).cuda().view(torch.bfloat16)
    dB = torch.from_numpy(Bb.view(np.int16)).cuda().view(torch.bfloat16)
    C = binding.gemm_bf16(dA, dB)
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = split_round_positions(M, N, np.random.default_rng(5))
    want = oracle.gemm_bf16_at(Ab, Bb, rows, cols)
    assert bits_equal(C[rows, cols], want)


@pytest.mark.parametrize("shape", [(256, 256, 256), (1024, 1024, 1024), (1000, 1003, 997),
                                   (129, 65, 24)], ids=lambda s: "x".join(map(str, s)))
def test_bf16_integer_pattern_exact(shape):
    M, N, K = shape
    A, B = inputs.integer_pattern(M, N, K)
    Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    C = run_bf16(Ab, Bb)
    want = oracle.gemm_bf16(Ab, Bb)
    assert bits_equal(C, want)


def test_bf16_dyadic_exact_misaligned():
    A = inputs.dyadic(300, 77, seed=21, denom=16, span=64)
    B = inputs.dyadic(77, 190, seed=22, denom=16, span=64)
    Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    for shift in (0, 1, 3):
        assert bits_equal(run_bf16(Ab, Bb, shift), oracle.gemm_bf16(Ab, Bb))


def test_bf16_ragged_tolerance():
    M, N, K = 1000, 1003, 997
    Ab, Bb = inputs.uniform_bf16(M, K, 1003), inputs.uniform_bf16(K, N, 2003)
    C = run_bf16(Ab, Bb)
    assert float(np.max(np.abs(C - oracle.gemm_bf16(Ab, Bb)))) <= tolerance(Ab, Bb)


def small_shapes():
    edge = [1, 2, 3, 7, 8, 9, 16, 31, 63, 64, 65, 127, 128, 129, 200, 257]
    rng = np.random.default_rng(4321)
    shapes = {(1, 1, 1), (1, 1, 257), (257, 1, 1), (1, 257, 1), (128, 256, 64), (129, 257, 72)}
    while len(shapes) < 40:
        shapes.add(tuple(int(x) for x in rng.choice(edge, 3)))
    return sorted(shapes)


@pytest.mark.parametrize("shift", [0, 1], ids=["aligned", "misaligned"])
@pytest.mark.parametrize("shape", small_shapes(), ids=lambda s: "x".join(map(str, s)))
def test_bf16_small_shapes(shape, shift):
    """K % 8 != 0 or a misaligned A takes the padded-A path; the others read A in place."""
    M, N, K = shape
    Ab, Bb = inputs.uniform_bf16(M, K, 31 + M), inputs.uniform_bf16(K, N, 37 + N)
    C = run_bf16(Ab, Bb, shift)
    assert float(np.max(np.abs(C - oracle.gemm_bf16(Ab, Bb)))) <= tolerance(Ab, Bb)


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (8192, 8192, 8192), (16384, 16384, 32),
                                   (8192, 8192, 64), (512, 512, 512), (256, 256, 65536),
                                   (130, 70, 20000), (4096, 4096, 16384), (4096, 4096, 16448)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_large_sampled(shape):
    """Full-size shapes (the benchmarked 4096^3 among them) on sampled outputs; 4096^2 x 16384
    is the longest K the 256 x 512 tiles take (all of K summed in TMEM), 16448 the first that
    goes back to chunked sums."""
    M, N, K = shape
    Ab, Bb = inputs.uniform_bf16(M, K, 1005), inputs.uniform_bf16(K, N, 2005)
    C = binding.gemm_bf16(bf16_tensor(Ab), bf16_tensor(Bb))
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = sample_positions(M, N, np.random.default_rng(M + K))
    ref = oracle.gemm_bf16_at(Ab, Bb, rows, cols)
    assert float(np.max(np.abs(C[rows, cols] - ref))) <= tolerance(Ab, Bb)


def edge_positions(M, N, rng):
    """Every element of the last 200 rows and of the last 520 columns (ragged 256 x 512 pair
    tiles at the bottom and right edges), the first row and column, and random positions."""
    rr, cc = np.meshgrid(np.arange(M - 200, M), np.arange(N), indexing="ij")
    r2, c2 = np.meshgrid(np.arange(M), np.arange(N - 520, N), indexing="ij")
    rows = [rr.ravel(), r2.ravel(), np.zeros(N, np.int64), np.arange(M), rng.integers(0, M, 4096)]
    cols = [cc.ravel(), c2.ravel(), np.arange(N), np.zeros(M, np.int64), rng.integers(0, N, 4096)]
    return np.concatenate(rows), np.concatenate(cols)


@pytest.mark.parametrize("kind", ["integer", "uniform"])
def test_bf16_wide_tiles_ragged_edges(kind):
    """2500 x 2000 x 3000 runs 256 x 512 pair tiles (80 of them) with partial tiles at the
    bottom (2500 = 9 x 256 + 196) and the right (2000 = 3 x 512 + 464) and a partial last
    k block (K = 3000): integer operands must give the definition's bits, uniform ones stay
    within the tolerance."""
    M, N, K = 2500, 2000, 3000
    if kind == "integer":
        A, B = inputs.integer_pattern(M, N, K)
        Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    else:
        Ab, Bb = inputs.uniform_bf16(M, K, 1007), inputs.uniform_bf16(K, N, 2007)
    C = binding.gemm_bf16(bf16_tensor(Ab), bf16_tensor(Bb))
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = edge_positions(M, N, np.random.default_rng(9))
    ref = oracle.gemm_bf16_at(Ab, Bb, rows, cols)
    if kind == "integer":
        assert bits_equal(C[rows, cols], ref)
    else:
        assert float(np.max(np.abs(C[rows, cols] - ref))) <= tolerance(Ab, Bb)


def test_bf16_nan_and_inf_propagate():
    M, N, K = 130, 140, 96
    A = inputs.dyadic(M, K, seed=41, denom=4, span=8)
    B = np.abs(inputs.dyadic(K, N, seed=42, denom=4, span=8)) + np.float32(0.25)  # all > 0
    Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    Ab[5, 17] = BF16_NAN
    Ab[77, 90] = 0x7F80  # +inf; every B entry is positive, so row 77 is +inf
    C = run_bf16(Ab, Bb)
    assert np.all(np.isnan(C[5])) and np.all(np.isposinf(C[77]))
    rest = np.ones(M, bool)
    rest[[5, 77]] = False
    assert bits_equal(C[rest], oracle.gemm_bf16(Ab, Bb)[rest])


def test_bf16_contract_checks():
    M, N, K = 64, 48, 40
    dA = torch.zeros((M * K + 8,), dtype=torch.int16, device="cuda")
    dB = torch.zeros((K * N + 8,), dtype=torch.int16, device="cuda")
    dC = torch.full((M * N,), 7.0, device="cuda")
    need = binding.t2s_gemm_bf16_f32_workspace_size(M, N, K)
    assert need > 0 and binding.t2s_gemm_bf16_f32_workspace_size(-1, N, K) == 0
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    f = binding.t2s_gemm_bf16_f32
    a, b, c, w = dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), ws.data_ptr()
    assert f(M, N, K, a, b, c, 0, need, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, a, b, c, w, need - 1, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, a, b, c, w + 16, need, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, a + 1, b, c, w, need, s) == binding.T2S_ERR_INVALID  # odd address
    assert f(M, N, K, a, b, c + 2, w, need, s) == binding.T2S_ERR_INVALID  # C not 4-aligned
    assert f(M, N, K, a, b, a, w, need, s) == binding.T2S_ERR_INVALID  # C == A
    assert f(-1, N, K, a, b, c, w, need, s) == binding.T2S_ERR_INVALID
    assert f(0, N, K, 0, b, 0, 0, 0, s) == binding.T2S_OK  # nothing to do
    assert f(M, N, 0, 0, 0, c, w, need, s) == binding.T2S_OK  # K = 0: C = +0.0
    torch.cuda.synchronize()
    assert torch.all(dC == 0) and not torch.any(torch.signbit(dC))
    assert f(M, N, K, a, b, c, w, need, s) == binding.T2S_OK
    assert binding.t2s_device_status(s) == binding.T2S_OK


@pytest.mark.parametrize("shape", [(128, 64, 64), (300, 200, 130), (129, 8, 1000), (77, 72, 37),
                                   (513, 392, 520), (256, 264, 4096), (1000, 1000, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_b_read_in_place(shape):
    """N % 8 == 0 and B 16-byte aligned: B is read in place as MN-major atoms (no transpose);
    ragged N leaves a partly empty last 64-column box."""
    M, N, K = shape
    Ab, Bb = inputs.uniform_bf16(M, K, 61 + M), inputs.uniform_bf16(K, N, 67 + N)
    C = run_bf16(Ab, Bb)
    assert float(np.max(np.abs(C - oracle.gemm_bf16(Ab, Bb)))) <= tolerance(Ab, Bb)
    A, B = inputs.integer_pattern(M, N, K)
    Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    assert bits_equal(run_bf16(Ab, Bb), oracle.gemm_bf16(Ab, Bb))


@pytest.mark.parametrize("shape", [(389, 512, 256), (129, 256, 136), (300, 64, 200),
                                   (1280, 1024, 2048), (3 * 128, 320, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_paired_tiles(shape):
    """M > 128 with B read in place runs clusters of two CTAs on vertically adjacent tiles that
    share B: an odd number of tile rows leaves the last pair's second tile beyond M."""
    M, N, K = shape
    Ab, Bb = inputs.uniform_bf16(M, K, 71 + M), inputs.uniform_bf16(K, N, 73 + N)
    C = run_bf16(Ab, Bb)
    assert float(np.max(np.abs(C - oracle.gemm_bf16(Ab, Bb)))) <= tolerance(Ab, Bb)
    A, B = inputs.integer_pattern(M, N, K)
    Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    assert bits_equal(run_bf16(Ab, Bb), oracle.gemm_bf16(Ab, Bb))


@pytest.mark.parametrize("shape", [(512, 512, 192), (300, 256, 72), (640, 512, 4160), (256, 768, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_paired_deep_k_blocks(shape):
    """256-wide pair tiles stage 128-deep K blocks: K not a multiple of 128 ends in a half-empty
    block (zeros from TMA), and K < 64 in a single partly filled one."""
    M, N, K = shape
    Ab, Bb = inputs.uniform_bf16(M, K, 91 + M), inputs.uniform_bf16(K, N, 93 + N)
    C = run_bf16(Ab, Bb)
    assert float(np.max(np.abs(C - oracle.gemm_bf16(Ab, Bb)))) <= tolerance(Ab, Bb)
    A, B = inputs.integer_pattern(M, N, K)
    Ab, Bb = inputs.to_bf16_bits(A), inputs.to_bf16_bits(B)
    assert bits_equal(run_bf16(Ab, Bb), oracle.gemm_bf16(Ab, Bb))
