"""Concurrent use of the library (GPU): several host threads, each with its own stream, call
the entry points at once; every result must be the one a lone call gives (the product kernel's
bits, the host pipeline's bits), so no state is shared between calls by accident."""
from __future__ import annotations

import threading

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


def test_threads_on_own_streams_match_lone_calls():
    shapes = [(700, 900, 513), (1024, 1024, 256), (333, 257, 1000), (2048, 512, 128)]
    data = []
    for t, (M, N, K) in enumerate(shapes):
        A, B = inputs.uniform_pair(M, N, K, 20 + t)
        data.append((A, B, oracle.sgemm(A, B, oracle.FMA)))
    results = [None] * (2 * len(shapes))
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            A, B, _ = data[i % len(shapes)]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
                for _ in range(3):
                    C = binding.gemm(dA, dB, stream=s.cuda_stream)
                s.synchronize()
                results[i] = C.cpu().numpy()
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(results))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert binding.device_status() == binding.T2S_OK
    for i, C in enumerate(results):
        want = data[i % len(shapes)][2]
        assert np.array_equal(C.view(np.uint32), want.view(np.uint32)), i


def test_host_pipeline_from_two_threads():
    M, N, K = 2048, 1024, 512
    pairs = [inputs.uniform_pair(M, N, K, 30 + t) for t in range(2)]
    want = [oracle.sgemm(A, B, oracle.FMA) for A, B in pairs]
    out = [None, None]
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            A, B = pairs[i]
            hA = torch.from_numpy(A).pin_memory()
            hB = torch.from_numpy(B).pin_memory()
            hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
            dA = torch.empty((M, K), device="cuda")
            dB = torch.empty((K, N), device="cuda")
            dC = torch.empty((M, N), device="cuda")
            s = torch.cuda.Stream()
            for _ in range(2):
                rc = binding.t2s_gemm_f32_host(M, N, K, hA.data_ptr(), hB.data_ptr(), hC.data_ptr(),
                                               dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                                               s.cuda_stream)
                assert rc == binding.T2S_OK
            s.synchronize()
            out[i] = hC.numpy().copy()
        except Exception as e:
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i in range(2):
        assert np.array_equal(out[i].view(np.uint32), want[i].view(np.uint32)), i
