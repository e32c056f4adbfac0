"""Parity of the CUDA kernels with the CPU oracle (GPU tests, through the C ABI).

Bars:
* the FFMA kernels (product, naive, smem32) use one IEEE fused multiply-add per k in
  ascending k, so they must equal the oracle's fused reading bit for bit on every
  input; on the integer-pattern inputs, where every operation is exact, they must
  also equal the two-rounding reading bit for bit;
* against the two-rounding reading (the literal C statement), the bound is
  max |C_gpu - C_oracle| <= 1e-6 * K * max|a| * max|b|;
* the 3xTF32 tensor-core kernel must meet that same bound against both readings,
  and be exact on the integer pattern.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from roofline_driven_tiling_gb300 import binding, inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FFMA_KERNELS = ("ffma", "naive", "smem32")
GUARD = 64  # canary floats on each side of every buffer
C_SENTINEL = np.float32(-12345.678)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    assert binding.device_status() == binding.T2S_OK


class Guarded:
    """A device copy of a matrix with NaN canaries (inputs) or sentinels (output)
    on both sides; `shift` floats of extra offset make the data 4-byte aligned only."""

    def __init__(self, x: np.ndarray, fill: float, shift: int = 0):
        n = x.size
        self.shape = x.shape
        self.n = n
        self.start = GUARD + shift
        self.buf = torch.full((n + 2 * GUARD + shift,), float(fill), dtype=torch.float32,
                              device="cuda")
        if n:
            self.buf[self.start:self.start + n] = torch.from_numpy(np.ascontiguousarray(x).ravel()).cuda()

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + 4 * self.start

    def data(self) -> np.ndarray:
        return self.buf[self.start:self.start + self.n].cpu().numpy().reshape(self.shape)

    def guards_intact(self, fill: float) -> bool:
        host = self.buf.cpu().numpy()
        lo, hi = host[:self.start], host[self.start + self.n:]
        if np.isnan(fill):
            return bool(np.all(np.isnan(lo)) and np.all(np.isnan(hi)))
        return bool(np.all(lo == fill) and np.all(hi == fill))


def run(kernel: str, A: np.ndarray, B: np.ndarray, shift: int = 0, stream=None):
    """Runs one kernel through the C ABI on guarded device buffers; returns C (host)."""
    M, K = A.shape
    N = B.shape[1]
    dA = Guarded(A, np.nan, shift)
    dB = Guarded(B, np.nan, shift)
    dC = Guarded(np.full((M, N), C_SENTINEL, np.float32), C_SENTINEL, shift)
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    if kernel == "tf32x3":
        need = binding.t2s_gemm_f32_tf32x3_workspace_size(M, N, K)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        rc = binding.t2s_gemm_f32_tf32x3(M, N, K, dA.ptr, dB.ptr, dC.ptr, ws.data_ptr(),
                                         ws.numel(), s)
    else:
        rc = getattr(binding, binding.KERNELS[kernel])(M, N, K, dA.ptr, dB.ptr, dC.ptr, s)
    assert rc == binding.T2S_OK, binding.status_string(rc)
    assert binding.t2s_device_status(s) == binding.T2S_OK
    assert dA.guards_intact(np.nan) and dB.guards_intact(np.nan)
    assert dC.guards_intact(C_SENTINEL), "write outside C"
    return dC.data()


def bits_equal(x: np.ndarray, y: np.ndarray) -> bool:
    return np.array_equal(x.view(np.uint32), y.view(np.uint32))


def mismatch(x: np.ndarray, y: np.ndarray) -> str:
    bad = np.argwhere(x.view(np.uint32) != y.view(np.uint32))
    if bad.size == 0:
        return "equal"
    i = tuple(bad[0])
    return "%d elements differ; first at %s: %r vs %r" % (len(bad), i, x[i], y[i])


def tolerance(A: np.ndarray, B: np.ndarray) -> float:
    K = A.shape[1]
    return 1e-6 * K * float(np.max(np.abs(A))) * float(np.max(np.abs(B)))


# ------------------------------------------------------------------ the workloads
@pytest.mark.parametrize("kernel", FFMA_KERNELS)
@pytest.mark.parametrize("n", [256, 1024])
def test_integer_pattern_bit_exact(kernel, n):
    A, B = inputs.integer_pattern(n, n, n)
    C = run(kernel, A, B)
    for mode in (oracle.FMA, oracle.MUL_ADD):
        want = oracle.sgemm(A, B, mode)
        assert bits_equal(C, want), mismatch(C, want)


@pytest.mark.parametrize("kernel", FFMA_KERNELS)
def test_constant_inputs_1024(kernel):
    n = 1024
    A, B = inputs.constant(n, n, n)
    C = run(kernel, A, B)
    want = oracle.sgemm_rows(A, B, 0, 8, oracle.FMA)[0, 0]
    assert np.all(C == want)  # every entry is the same sum
    exact = n * 0.5 * float(np.float32(0.4))
    gamma = n * 2.0 ** -24 / (1 - n * 2.0 ** -24)
    assert abs(float(C[0, 0]) - exact) <= gamma * exact  # closed form 0.2 K within gamma_K


@pytest.mark.parametrize("kernel", FFMA_KERNELS)
def test_ragged_1000x1003x997(kernel):
    M, N, K = 1000, 1003, 997
    A, B = inputs.uniform_pair(M, N, K, 3)
    C = run(kernel, A, B)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert bits_equal(C, want), mismatch(C, want)
    lit = oracle.sgemm(A, B, oracle.MUL_ADD)
    assert float(np.max(np.abs(C - lit))) <= tolerance(A, B)


def sample_positions(M, N, rng, n_random=4096):
    rows = [0, M - 1, M // 2]
    cols = [0, N - 1, N // 2]
    r = [np.full(N, i) for i in rows] + [np.arange(M) for _ in cols]
    c = [np.arange(N) for _ in rows] + [np.full(M, j) for j in cols]
    r.append(rng.integers(0, M, n_random))
    c.append(rng.integers(0, N, n_random))
    return np.concatenate(r), np.concatenate(c)


def check_sampled(C, A, B, seed=0):
    M, N = C.shape
    rows, cols = sample_positions(M, N, np.random.default_rng(seed))
    want = oracle.sgemm_at(A, B, rows, cols, oracle.FMA)
    got = C[rows, cols]
    assert bits_equal(got, want), mismatch(got, want)
    lit = oracle.sgemm_at(A, B, rows, cols, oracle.MUL_ADD)
    assert float(np.max(np.abs(got - lit))) <= tolerance(A, B)


def test_headline_4096_every_element():
    """The benchmarked workload (4096^3, uniform, config 4) in the benchmarked launch (whole
    rounds of 256 x 128 tiles, then the 64 x 64 tail), against the oracle's fused
    multiply-add reading on every one of the 16.8 M elements, bit for bit (the oracle takes
    about 11 s on 16 host cores), and within the tolerance of the two-rounding reading on a
    sample."""
    A, B = inputs.uniform_pair(4096, 4096, 4096, 4)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = binding.gemm(dA, dB).cpu().numpy()
    assert binding.device_status() == binding.T2S_OK
    assert np.all(np.isfinite(C))
    want = oracle.sgemm(A, B, oracle.FMA)
    assert bits_equal(C, want), mismatch(C, want)
    check_sampled(C, A, B)


@pytest.mark.parametrize("shape", inputs.SWEEP, ids=lambda s: "x".join(map(str, s)))
def test_sweep_sampled(shape):
    M, N, K = shape
    A, B = inputs.uniform_pair(M, N, K, 5)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = binding.gemm(dA, dB).cpu().numpy()
    assert binding.device_status() == binding.T2S_OK
    check_sampled(C, A, B, seed=M + N + K)


# ------------------------------------------------------------------ edges
def small_shapes():
    edge = [1, 2, 3, 4, 5, 7, 8, 31, 32, 33, 63, 64, 65, 127, 128, 129, 191, 257]
    rng = np.random.default_rng(1234)
    shapes = {(1, 1, 1), (1, 1, 257), (257, 1, 1), (1, 257, 1), (129, 129, 129), (64, 64, 64),
              (128, 128, 32), (128, 128, 33), (65, 300, 31)}
    while len(shapes) < 90:
        shapes.add(tuple(int(x) for x in rng.choice(edge, 3)))
    return sorted(shapes)


@pytest.mark.parametrize("shift", [0, 1], ids=["aligned", "misaligned"])
@pytest.mark.parametrize("shape", small_shapes(), ids=lambda s: "x".join(map(str, s)))
def test_small_ragged_shapes(shape, shift):
    M, N, K = shape
    A = inputs.uniform(M, K, 7 + M)
    B = inputs.uniform(K, N, 9 + N)
    want = oracle.sgemm(A, B, oracle.FMA)
    for kernel in FFMA_KERNELS if shift == 0 else ("ffma",):
        C = run(kernel, A, B, shift=shift)
        assert bits_equal(C, want), "%s: %s" % (kernel, mismatch(C, want))


def test_misaligned_equals_aligned():
    """The cp.async load path (4-byte aligned pointers) gives the TMA path's bits."""
    A, B = inputs.uniform_pair(384, 256, 512, 11)
    assert bits_equal(run("ffma", A, B, shift=0), run("ffma", A, B, shift=1))


@pytest.mark.parametrize("kernel", FFMA_KERNELS)
def test_k_zero_writes_positive_zero(kernel):
    A = np.zeros((33, 0), np.float32)
    B = np.zeros((0, 17), np.float32)
    C = run(kernel, A, B)
    assert np.all(C.view(np.uint32) == 0)


def test_non_default_stream():
    A, B = inputs.uniform_pair(520, 260, 132, 12)
    s = torch.cuda.Stream()
    C = run("ffma", A, B, stream=s)
    assert bits_equal(C, oracle.sgemm(A, B, oracle.FMA))


def test_bounded_wait_reports_timeout():
    """A barrier nothing arrives on: the kernel gives up, records the timeout and the
    context stays usable."""
    s = torch.cuda.current_stream().cuda_stream
    assert binding.t2s_selftest_wait_timeout(2_000_000, s) == binding.T2S_OK
    assert binding.t2s_device_status(s) == binding.T2S_ERR_TIMEOUT
    assert binding.t2s_device_status(s) == binding.T2S_OK  # read clears it
    A, B = inputs.uniform_pair(64, 64, 64, 13)
    assert bits_equal(run("ffma", A, B), oracle.sgemm(A, B, oracle.FMA))


# ------------------------------------------------------------------ 3xTF32 tensor-core kernel
@pytest.mark.parametrize("n", [256, 1024])
def test_tf32x3_integer_pattern_exact(n):
    """Small integers are exact in TF32 (the small parts are zero) and every sum is exact."""
    A, B = inputs.integer_pattern(n, n, n)
    C = run("tf32x3", A, B)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert bits_equal(C, want), mismatch(C, want)


def test_tf32x3_ragged_tolerance():
    M, N, K = 1000, 1003, 997
    A, B = inputs.uniform_pair(M, N, K, 3)
    C = run("tf32x3", A, B)
    for mode in (oracle.FMA, oracle.MUL_ADD):
        ref = oracle.sgemm(A, B, mode)
        assert float(np.max(np.abs(C - ref))) <= tolerance(A, B)


def test_tf32x3_constant_closed_form():
    n = 1024
    A, B = inputs.constant(n, n, n)
    C = run("tf32x3", A, B)
    exact = n * 0.5 * float(np.float32(0.4))
    gamma = n * 2.0 ** -24 / (1 - n * 2.0 ** -24)
    assert float(np.max(np.abs(C.astype(np.float64) - exact))) <= 2 * gamma * exact


def test_tf32x3_headline_sampled():
    A, B = inputs.uniform_pair(4096, 4096, 4096, 4)
    C = binding.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), kernel="tf32x3")
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = sample_positions(4096, 4096, np.random.default_rng(4))
    got = C[rows, cols]
    for mode in (oracle.FMA, oracle.MUL_ADD):
        ref = oracle.sgemm_at(A, B, rows, cols, mode)
        assert float(np.max(np.abs(got - ref))) <= tolerance(A, B)


@pytest.mark.parametrize("shape", small_shapes()[::3], ids=lambda s: "x".join(map(str, s)))
def test_tf32x3_small_shapes(shape):
    M, N, K = shape
    A = inputs.uniform(M, K, 17 + M)
    B = inputs.uniform(K, N, 19 + N)
    C = run("tf32x3", A, B)
    ref = oracle.sgemm(A, B, oracle.MUL_ADD)
    assert float(np.max(np.abs(C - ref))) <= tolerance(A, B)


@pytest.mark.parametrize("shift", [1])
def test_tf32x3_misaligned_inputs(shift):
    A, B = inputs.uniform_pair(257, 131, 67, 14)
    C = run("tf32x3", A, B, shift=shift)
    assert float(np.max(np.abs(C - oracle.sgemm(A, B, oracle.MUL_ADD)))) <= tolerance(A, B)


@pytest.mark.parametrize("shift", [0, 1], ids=["aligned", "misaligned"])
def test_tf32x3_special_values(shift):
    """NaNs (quiet, and one whose payload sits only in the 13 low mantissa bits that TF32
    drops), infinities, signed zeros and subnormal operands. A NaN in row i of A makes row i
    of C NaN, as in the definition; an infinity makes its row non-finite (it stays infinite,
    or a correction term multiplies it by the zero small part of an exactly representable
    operand); every other element is finite and within the tolerance."""
    M, N, K = 131, 136, 96
    A, B = inputs.uniform_pair(M, N, K, 17)
    tiny = np.float32(1.4e-45)
    A[10, 3], A[20, 7], B[5, 9], B[6, 11] = np.float32(-0.0), tiny, np.float32(1e-40), -tiny
    A[3, 5] = np.frombuffer(np.uint32(0x7F800001).tobytes(), dtype=np.float32)[0]  # NaN
    A[40, 50] = np.float32(np.nan)
    A[60, 2] = np.float32(np.inf)
    A[70, 80] = np.float32(-np.inf)
    C = run("tf32x3", A, B, shift=shift)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert np.all(np.isnan(C[[3, 40]])) and np.all(np.isnan(want[[3, 40]]))
    assert not np.any(np.isfinite(C[[60, 70]]))
    rest = np.ones(M, bool)
    rest[[3, 40, 60, 70]] = False
    assert np.all(np.isfinite(C[rest]))
    assert float(np.max(np.abs(C[rest] - want[rest]))) <= tolerance(A[rest], B)


@pytest.mark.parametrize("operand", ["A", "B"])
def test_tf32x3_finite_operands_next_to_flt_max(operand):
    """Finite operands within half a TF32 ulp of FLT_MAX (which round up to infinity in TF32)
    and a few more of the largest binary32 values, in one operand; the other operand is
    scaled by 2^-24 so that every element of the definition stays finite. The split must keep
    them finite: the result is finite everywhere and within the tolerance of the oracle."""
    M, N, K = 131, 136, 96
    A, B = inputs.uniform_pair(M, N, K, 23)
    big = np.frombuffer(np.array([0x7F7FFFFF, 0xFF7FFFFF, 0x7F7FF000, 0xFF7FF800, 0x7F7FEFFF,
                                  0x7F7FC99E], dtype=np.uint32).tobytes(), dtype=np.float32)
    if operand == "A":
        B *= np.float32(2.0 ** -24)
        pos = [(3, 5), (3, 6), (40, 50), (60, 2), (70, 80), (130, 95)]
        for (i, k), v in zip(pos, big):
            A[i, k] = v
    else:
        A *= np.float32(2.0 ** -24)
        pos = [(5, 3), (6, 3), (50, 40), (2, 60), (80, 70), (95, 135)]
        for (k, j), v in zip(pos, big):
            B[k, j] = v
    want = oracle.sgemm(A, B, oracle.MUL_ADD)
    assert np.all(np.isfinite(want))
    C = run("tf32x3", A, B)
    assert np.all(np.isfinite(C)), "a finite operand near FLT_MAX gave a non-finite result"
    assert float(np.max(np.abs(C - want))) <= tolerance(A, B)


@pytest.mark.parametrize("shape", [(4000, 4100, 520), (4096, 4096, 1024), (1324, 2500, 300)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32x3_pair_tiles(shape):
    """Shapes the 3xTF32 dispatch runs on CTA pairs (256-row tiles, cta_group::2 MMAs, each CTA
    staging half of the B planes): ragged M (the last pair's second CTA holds rows past M, or
    none), ragged N (a partial last tile of 224 or 256 columns), K not a multiple of the
    32-value padding. Checked on whole rows and columns at the edges and on random elements
    against both readings of the oracle, within the FP32 tolerance."""
    M, N, K = shape
    A, B = inputs.uniform_pair(M, N, K, 29)
    C = run("tf32x3", A, B)
    assert np.all(np.isfinite(C))
    rows, cols = sample_positions(M, N, np.random.default_rng(M + N + K), n_random=8192)
    for mode in (oracle.FMA, oracle.MUL_ADD):
        want = oracle.sgemm_at(A, B, rows, cols, mode)
        assert float(np.max(np.abs(C[rows, cols] - want))) <= tolerance(A, B)


def test_tf32x3_workspace_checks():
    M, N, K = 64, 64, 64
    dA = torch.zeros((M, K), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    dC = torch.zeros((M, N), device="cuda")
    need = binding.t2s_gemm_f32_tf32x3_workspace_size(M, N, K)
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    f = binding.t2s_gemm_f32_tf32x3
    assert f(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), 0, need, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), ws.data_ptr(), need - 1, s) == \
        binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), ws.data_ptr() + 4, need, s) == \
        binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), ws.data_ptr(), need, s) == binding.T2S_OK
    assert binding.t2s_device_status(s) == binding.T2S_OK


@pytest.mark.parametrize("shape", inputs.SWEEP + [(256, 256, 65536), (130, 70, 20000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tf32x3_sweep_and_long_k_sampled(shape):
    """The tolerance must hold at every sweep shape and for long K, where an accumulation
    that does not round to nearest drifts further with every added term."""
    M, N, K = shape
    A, B = inputs.uniform_pair(M, N, K, 5)
    C = binding.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), kernel="tf32x3")
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = sample_positions(M, N, np.random.default_rng(M + K))
    got = C[rows, cols]
    for mode in (oracle.FMA, oracle.MUL_ADD):
        ref = oracle.sgemm_at(A, B, rows, cols, mode)
        assert float(np.max(np.abs(got - ref))) <= tolerance(A, B)



# ------------------------------------------------------------------ host-memory entry point
@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (1000, 1003, 997), (1537, 260, 129),
                                   (3, 5, 0), (600, 17, 33), (2100, 130, 1001), (2048, 96, 600),
                                   (3072, 64, 4096), (1500, 700, 2051), (2500, 1000, 3000),
                                   (1100, 333, 2100), (512, 512, 9000), (3000, 2900, 2600),
                                   (1024, 1024, 2600)],
                         ids=lambda s: "x".join(map(str, s)))
def test_host_pipeline_equals_device_entry(shape):
    """Copy-overlapped product of host matrices, by row blocks or by K chunks that resume from
    the sums stored in C (4096^3, 3072 x 64 x 4096 and the last six shapes; 4096^3 and
    3000 x 2900 x 2600 have the shorter edge chunks of products with at least 2^23 outputs, and
    1024 x 1024 x 2600 runs chunks that are not multiples of 64 on the tile whose whole-K
    launches take 64-deep K blocks): the bits of t2s_gemm_f32."""
    M, N, K = shape
    A = inputs.uniform(M, K, 31 + M)
    B = inputs.uniform(K, N, 37 + N)
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.full((M, N), float("nan")).pin_memory()
    dA = torch.empty((M, K), device="cuda")
    dB = torch.empty((K, N), device="cuda")
    dC = torch.empty((M, N), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = binding.t2s_gemm_f32_host(M, N, K, hA.data_ptr(), hB.data_ptr(), hC.data_ptr(),
                                   dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), s)
    assert rc == binding.T2S_OK, binding.status_string(rc)
    assert binding.t2s_device_status(s) == binding.T2S_OK
    got = hC.numpy()
    if K == 0:
        assert np.all(got.view(np.uint32) == 0)
        return
    want = binding.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()).cpu().numpy()
    assert bits_equal(got, want), mismatch(got, want)
    rows, cols = sample_positions(M, N, np.random.default_rng(7))
    ref = oracle.sgemm_at(A, B, rows, cols, oracle.FMA)
    assert bits_equal(got[rows, cols], ref)


# ------------------------------------------------------------------ special values
def special_inputs(M, N, K, seed):
    """Uniform values with infinities, NaNs, signed zeros, subnormals and large magnitudes
    planted at random positions."""
    rng = np.random.default_rng(seed)
    A = inputs.uniform(M, K, seed)
    B = inputs.uniform(K, N, seed + 1)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-40, -3e-39, 1e30, -2e30,
                         np.float32(1.4e-45)], dtype=np.float32)
    for X in (A, B):
        idx = rng.choice(X.size, size=max(1, X.size // 200), replace=False)
        X.ravel()[idx] = rng.choice(specials, size=idx.size)
    return A, B


@pytest.mark.parametrize("kernel", FFMA_KERNELS)
@pytest.mark.parametrize("shift", [0, 1], ids=["aligned", "misaligned"])
def test_special_values_match_fma_oracle(kernel, shift):
    """IEEE fused multiply-adds in the oracle's order give the same infinities, signed
    zeros, subnormal results and NaN positions; finite results agree bit for bit."""
    if kernel != "ffma" and shift:
        pytest.skip("alignment only selects a load path of the product kernel")
    M, N, K = 131, 257, 203
    A, B = special_inputs(M, N, K, 77)
    C = run(kernel, A, B, shift=shift)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert np.array_equal(np.isnan(C), np.isnan(want))
    keep = ~np.isnan(want)
    assert bits_equal(C[keep], want[keep]), mismatch(C[keep], want[keep])


# ------------------------------------------------------------------ vector add (memory roof)
@pytest.mark.parametrize("n", [1, 7, 8, 9, 31, 1000, 4099, 1 << 20, (1 << 22) + 13])
@pytest.mark.parametrize("shift", [0, 1, 4], ids=["align32", "align4", "align16"])
def test_vector_add_matches_oracle(n, shift):
    x = inputs.uniform(1, n, 41 + n).ravel()
    y = inputs.uniform(1, n, 43 + n).ravel()
    if n > 8:
        x[3], y[5], x[7], y[7] = np.inf, np.nan, -0.0, -0.0
    dx, dy = Guarded(x, np.nan, shift), Guarded(y, np.nan, shift)
    dz = Guarded(np.full(n, C_SENTINEL, np.float32), C_SENTINEL, shift)
    s = torch.cuda.current_stream().cuda_stream
    assert binding.t2s_vector_add_f32(n, dx.ptr, dy.ptr, dz.ptr, s) == binding.T2S_OK
    assert binding.t2s_device_status(s) == binding.T2S_OK
    assert dz.guards_intact(C_SENTINEL)
    got, want = dz.data(), oracle.vector_add(x, y)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    keep = ~np.isnan(want)
    assert bits_equal(got[keep], want[keep])


# ------------------------------------------------------------------ every product configuration
# One shape per configuration the dispatcher picks on a 152-SM GB300 (tile counts in the
# comments), each on the TMA path (aligned) and the cp.async path (K and N not multiples of 4).
DISPATCH_SHAPES = {
    "big_flat": (128, 131072, 288),        # 1024 tiles of 128^2 (7 per SM), K >= 256
    "huge_2560": (2560, 1920, 512),        # 150 tiles of 256 x 128: one round
    "huge_tail_2500": (2500, 2000, 512),   # 160 tiles of 256 x 128: 152, then 8 as 64 x 64
    "huge_tail_4096": (4096, 4096, 1024),  # 512 tiles of 256 x 128: 456, then 56 as 64 x 64
    "big_short_k": (3072, 3072, 128),      # 576 tiles of 128^2, K < 256
    "persistent_k32": (2560, 2560, 32),    # 400 tiles of 128^2, one K block (cp.async: 1)
    "pstore_k32": (8192, 4096, 32),        # 1024 tiles of 256 x 128, TMA stores (cp.async: 1)
    "pstore_k96": (3000, 4100, 96),        # 384 tiles of 256 x 128, ragged edges of C
    "tall88_1024": (1024, 3584, 1024),     # 448 tiles of 128 x 64: 8 x 8 per thread, pipelined
    "tall84_1152": (1152, 1024, 512),      # 144 tiles of 128 x 64, 8 warps of 8 x 4
    "wide74_1024": (1024, 1024, 512),      # 152 tiles of 56 x 128, 8 warps of 7 x 4
    "wide74_1792": (1792, 1792, 516),      # 448 tiles of 56 x 128, 2 stages, two CTAs per SM
    "big88_1536": (1536, 1536, 512),       # 144 tiles of 128 x 128, 8 warps of 8 x 8
    "small48_1280": (1280, 1280, 256),     # 400 tiles of 64 x 64, 4 x 8 per thread, 3 CTAs per SM
    "small48_640": (640, 700, 300),        # 110 tiles of 64 x 64
    "tiny24_384": (384, 384, 384),         # 144 tiles of 32 x 32, 2 x 4 per thread
}


# The plan code (t2s_gemm_f32_plan) each name stands for, by its prefix.
DISPATCH_PLANS = {"big_flat": 0, "big_short_k": 1, "tall88": 2, "small48": 3, "huge_tail": 5,
                  "huge": 4, "big88": 6, "tall84": 7, "persistent": 8, "wide74": 9, "tiny24": 10,
                  "pstore": 11}


@pytest.mark.parametrize("ragged", [False, True], ids=["tma", "cpasync"])
@pytest.mark.parametrize("name", sorted(DISPATCH_SHAPES))
def test_every_configuration(name, ragged):
    M, N, K = DISPATCH_SHAPES[name]
    if ragged:
        N, K = N - 1, K - 3
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        code = next(v for k, v in DISPATCH_PLANS.items() if name.startswith(k))
        assert binding.t2s_gemm_f32_plan(M, N, K, 152) == code
    A = inputs.uniform(M, K, 61 + M)
    B = inputs.uniform(K, N, 67 + N)
    C = run("ffma", A, B)
    rows, cols = sample_positions(M, N, np.random.default_rng(K))
    want = oracle.sgemm_at(A, B, rows, cols, oracle.FMA)
    assert bits_equal(C[rows, cols], want), mismatch(C[rows, cols], want)


@pytest.mark.parametrize("ragged", [False, True], ids=["tma", "cpasync"])
def test_huge_tail_every_element(ragged):
    """256 x 128 tiles in one whole round, the 8 tiles left over as 64 x 64 tiles in a second
    launch: every element, the ragged last tile row and column included, is the definition's."""
    M, N, K = 2500, 2000, 512
    if ragged:
        N, K = N - 1, K - 3
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert binding.t2s_gemm_f32_plan(M, N, K, 152) == 5
    A = inputs.uniform(M, K, 71)
    B = inputs.uniform(K, N, 73)
    C = run("ffma", A, B)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert bits_equal(C, want), mismatch(C, want)


def test_huge_tail_result_complete_for_next_launch():
    """The call is two launches on the caller's stream; work queued after it must see all of
    C. Here a second product reads the first one's C right away, twice in a row."""
    M, N, K, N2 = 2500, 2000, 512, 640
    A = inputs.uniform(M, K, 81)
    B = inputs.uniform(K, N, 83)
    B2 = inputs.uniform(N, N2, 85)
    dA, dB, dB2 = (torch.from_numpy(x).cuda() for x in (A, B, B2))
    s = torch.cuda.current_stream()
    for _ in range(2):
        C1 = binding.gemm(dA, dB, stream=s.cuda_stream)
        C2 = binding.gemm(C1, dB2, stream=s.cuda_stream)
    assert binding.device_status() == binding.T2S_OK
    want1 = oracle.sgemm(A, B, oracle.FMA)
    want2 = oracle.sgemm(want1, B2, oracle.FMA)
    assert bits_equal(C1.cpu().numpy(), want1)
    got2 = C2.cpu().numpy()
    assert bits_equal(got2, want2), mismatch(got2, want2)


# ------------------------------------------------------------------ split K
def run_splitk(A, B, splits, shift=0):
    M, K = A.shape
    N = B.shape[1]
    dA = Guarded(A, np.nan, shift)
    dB = Guarded(B, np.nan, shift)
    dC = Guarded(np.full((M, N), C_SENTINEL, np.float32), C_SENTINEL, shift)
    need = binding.t2s_gemm_f32_splitk_workspace_size(M, N, K, splits)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = binding.t2s_gemm_f32_splitk(M, N, K, dA.ptr, dB.ptr, dC.ptr, splits, ws.data_ptr(),
                                     ws.numel(), s)
    assert rc == binding.T2S_OK, binding.status_string(rc)
    assert binding.t2s_device_status(s) == binding.T2S_OK
    assert dC.guards_intact(C_SENTINEL)
    return dC.data()


@pytest.mark.parametrize("shape,splits", [((1024, 1024, 1024), 8), ((512, 512, 512), 0),
                                          ((256, 256, 4096), 0), ((1000, 1003, 997), 0),
                                          ((640, 640, 1280), 0), ((1000, 1003, 997), 4),
                                          ((300, 130, 1000), 3), ((64, 64, 2048), 64),
                                          ((129, 257, 33), 2)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_splitk_within_tolerance(shape, splits):
    M, N, K = shape
    A = inputs.uniform(M, K, 71 + M)
    B = inputs.uniform(K, N, 73 + N)
    C = run_splitk(A, B, splits)
    for mode in (oracle.FMA, oracle.MUL_ADD):
        ref = oracle.sgemm(A, B, mode)
        assert float(np.max(np.abs(C - ref))) <= tolerance(A, B)
    assert bits_equal(run_splitk(A, B, splits), C)  # deterministic


def test_splitk_one_chunk_is_the_product():
    A, B = inputs.uniform_pair(300, 200, 500, 15)
    assert bits_equal(run_splitk(A, B, 1), run("ffma", A, B))


def test_splitk_integer_pattern_exact_and_misaligned():
    A, B = inputs.integer_pattern(512, 512, 1024)
    C = run_splitk(A, B, 4)
    assert bits_equal(C, oracle.sgemm(A, B, oracle.FMA))  # exact sums in any order
    A, B = inputs.uniform_pair(257, 131, 999, 16)
    C = run_splitk(A, B, 5, shift=1)
    assert float(np.max(np.abs(C - oracle.sgemm(A, B, oracle.MUL_ADD)))) <= tolerance(A, B)


def test_splitk_workspace_checks():
    M, N, K = 256, 256, 1024
    dA = torch.zeros((M, K), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    dC = torch.zeros((M, N), device="cuda")
    need = binding.t2s_gemm_f32_splitk_workspace_size(M, N, K, 4)
    assert need == 4 * M * N * 4
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    f = binding.t2s_gemm_f32_splitk
    args = (M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), 4)
    assert f(*args, 0, need, s) == binding.T2S_ERR_WORKSPACE
    assert f(*args, ws.data_ptr(), need - 4, s) == binding.T2S_ERR_WORKSPACE
    assert f(*args, ws.data_ptr() + 4, need, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), 65, ws.data_ptr(), need, s) == \
        binding.T2S_ERR_INVALID
    assert f(*args, ws.data_ptr(), need, s) == binding.T2S_OK
    assert binding.t2s_device_status(s) == binding.T2S_OK


# ------------------------------------------------------------------ stream K
def run_streamk(A, B, shift=0):
    M, K = A.shape
    N = B.shape[1]
    dA = Guarded(A, np.nan, shift)
    dB = Guarded(B, np.nan, shift)
    dC = Guarded(np.full((M, N), C_SENTINEL, np.float32), C_SENTINEL, shift)
    need = binding.t2s_gemm_f32_streamk_workspace_size(M, N, K)
    ws = torch.full((max(need, 256) // 4,), float("nan"), device="cuda")  # stale partials show
    s = torch.cuda.current_stream().cuda_stream
    rc = binding.t2s_gemm_f32_streamk(M, N, K, dA.ptr, dB.ptr, dC.ptr, ws.data_ptr(),
                                      ws.numel() * 4, s)
    assert rc == binding.T2S_OK, binding.status_string(rc)
    assert binding.t2s_device_status(s) == binding.T2S_OK
    assert dA.guards_intact(np.nan) and dB.guards_intact(np.nan)
    assert dC.guards_intact(C_SENTINEL), "write outside C"
    return dC.data()


@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (2048, 2048, 2048), (1000, 1004, 996),
                                   (128, 128, 32), (256, 256, 8192), (1536, 1536, 1536),
                                   (130, 4100, 260), (2304, 640, 1024), (64, 64, 4),
                                   (5120, 2048, 128), (2048, 2432, 64), (5000, 2044, 100)],
                         ids=lambda s: "x".join(map(str, s)))
def test_streamk_within_tolerance(shape):
    """Equal shares of the tile x k-block space: tiles run whole by one CTA, shared by two or
    by many (long K, few tiles), a single iteration in all (128^3 / 32); with a data-parallel
    wave before the shared tiles (5120 x 2048: 640 tiles on 304 CTAs) and with a whole number
    of waves, all data-parallel (2048 x 2432: 304 tiles)."""
    M, N, K = shape
    A, B = inputs.uniform_pair(M, N, K, 8)
    C = run_streamk(A, B)
    assert np.all(np.isfinite(C))
    for mode in (oracle.FMA, oracle.MUL_ADD):
        ref = oracle.sgemm(A, B, mode)
        assert float(np.max(np.abs(C - ref))) <= tolerance(A, B)


def test_streamk_integer_exact_and_deterministic():
    A, B = inputs.integer_pattern(1536, 1024, 1024)
    C1 = run_streamk(A, B)
    C2 = run_streamk(A, B)
    assert bits_equal(C1, C2)
    want = oracle.sgemm(A, B, oracle.FMA)
    assert bits_equal(C1, want), mismatch(C1, want)


def test_streamk_headline_sampled():
    A, B = inputs.uniform_pair(4096, 4096, 4096, 4)
    C = binding.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), kernel="streamk")
    assert binding.device_status() == binding.T2S_OK
    C = C.cpu().numpy()
    rows, cols = sample_positions(4096, 4096, np.random.default_rng(44))
    for mode in (oracle.FMA, oracle.MUL_ADD):
        ref = oracle.sgemm_at(A, B, rows, cols, mode)
        assert float(np.max(np.abs(C[rows, cols] - ref))) <= tolerance(A, B)


def test_streamk_general_path_is_the_product():
    """K or N not a multiple of 4 (no TMA): the call runs the product kernel, bit-exact."""
    A, B = inputs.uniform_pair(300, 257, 131, 9)
    C = run_streamk(A, B)
    assert bits_equal(C, oracle.sgemm(A, B, oracle.FMA))
    A, B = inputs.uniform_pair(300, 256, 128, 9)
    C = run_streamk(A, B, shift=1)  # misaligned pointers: no TMA either
    assert bits_equal(C, oracle.sgemm(A, B, oracle.FMA))


def test_streamk_workspace_checks():
    M, N, K = 256, 256, 256
    dA = torch.zeros((M, K), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    dC = torch.zeros((M, N), device="cuda")
    need = binding.t2s_gemm_f32_streamk_workspace_size(M, N, K)
    assert need >= 2 * 128 * 128 * 4
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    f = binding.t2s_gemm_f32_streamk
    a, b, c, w = dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), ws.data_ptr()
    assert f(M, N, K, a, b, c, 0, need, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, a, b, c, w, need - 1, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, a, b, c, w + 4, need, s) == binding.T2S_ERR_WORKSPACE
    assert f(M, N, K, a, b, c, w, need, s) == binding.T2S_OK
    assert binding.t2s_device_status(s) == binding.T2S_OK
