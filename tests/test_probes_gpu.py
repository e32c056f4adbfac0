"""The throughput probes on the GPU, through the C ABI.

They supply the roofline's measured ceilings: the FP32 FMA pipe (packed fused multiply-adds
at the product kernels' occupancy) and the TF32 tensor pipe (tcgen05.mma kind::tf32 on
shared-memory operands). Their results are checked by what they compute: each FMA chain is
acc = 0.5 acc + 1, which reaches 2.0 exactly, so every thread's sum of 32 values is 64; the
MMA operands are zeros, so the accumulators are zero. Their rates must be positive and not
above the nominal unit counts (152 SMs x 128 lanes x 2 FLOP x 2.07 GHz for FP32; 2.25 PFLOP/s
x 1.1 / 2.25 for dense TF32, with room for clock and rounding). The store probe is checked by
the matrix it writes: every element of C holds the value, and the guard rows after C are untouched.
"""
from __future__ import annotations

import numpy as np
import pytest

from roofline_driven_tiling_gb300 import binding

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def timed_probe(kind, iters):
    n = binding.t2s_probe_outputs()
    assert n > 0
    out = torch.full((n,), float("nan"), device="cuda")
    stream = torch.cuda.current_stream()
    binding.probe(kind, iters, out.data_ptr(), stream.cuda_stream)  # warm-up
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    flops = binding.probe(kind, iters, out.data_ptr(), stream.cuda_stream)
    e.record(stream)
    torch.cuda.synchronize()
    assert binding.t2s_device_status(stream.cuda_stream) == binding.T2S_OK
    return flops / (s.elapsed_time(e) * 1e-3) / 1e12, out.cpu().numpy(), flops


def test_fp32_fma_probe():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rate, out, flops = timed_probe("fp32_fma", 1 << 14)
    threads = 2 * sms * 128
    assert flops == threads * (1 << 14) * 16 * 4
    assert np.all(out[:threads] == 64.0)
    nominal = sms * 128 * 2 * 2.07e9 / 1e12
    assert 0.3 * nominal < rate < 1.05 * nominal


def test_tf32_mma_probe():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rate, out, flops = timed_probe("tf32_mma", 1 << 11)
    assert flops == sms * (1 << 11) * 4 * 2 * 128 * 256 * 8
    assert np.all(out[:sms * 128] == 0.0)
    assert 100.0 < rate < 2250.0 * 1.1 / 2.25 * 1.3


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(1024, 1024), (512, 1152), (2304, 384)],
                         ids=lambda s: "%dx%d" % s)
def test_store_probe_writes_every_element(mode, shape):
    # 512 x 1152: one group of 2 tile rows; 2304 x 384: a group of 8 tile rows and one of 1.
    M, N = shape
    buf = torch.full((M + 4, N), float("nan"), device="cuda")
    stream = torch.cuda.current_stream()
    nbytes = binding.probe_store(M, N, buf.data_ptr(), mode, 3.5, stream.cuda_stream)
    torch.cuda.synchronize()
    assert binding.t2s_device_status(stream.cuda_stream) == binding.T2S_OK
    assert nbytes == 4 * M * N
    assert bool((buf[:M] == 3.5).all())
    assert bool(torch.isnan(buf[M:]).all())


def test_store_probe_rate():
    M = N = 8192
    C = torch.empty((M, N), device="cuda")
    stream = torch.cuda.current_stream()
    for mode in (0, 1):
        binding.probe_store(M, N, C.data_ptr(), mode, 1.0, stream.cuda_stream)  # warm-up
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        nbytes = binding.probe_store(M, N, C.data_ptr(), mode, 1.0, stream.cuda_stream)
        e.record(stream)
        torch.cuda.synchronize()
        rate = nbytes / (s.elapsed_time(e) * 1e-3) / 1e9
        # Positive and below the HBM3e nominal 7.9 TB/s with room (the matrix is above L2).
        assert 200.0 < rate < 9000.0, (mode, rate)
    assert bool((C == 1.0).all())
