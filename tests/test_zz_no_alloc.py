"""t2s_gemm_f32_tf32x3_noalloc: the 3xTF32 product for callers that cannot allocate.

Some callers cannot allocate device memory: a plugin whose host framework owns all device
memory through its own pool and budget, a latency-critical loop that cannot afford
cudaMalloc's implicit synchronisation, or C code with no device allocator. This entry
point keeps the split operands in a static device array inside the library instead of a
caller-provided workspace.

The GPU test compares it, through the C ABI, with the workspace entry point on the same
inputs, for two calls in a row with different shapes (so the second call runs on scratch
left by the first). Both run the same deterministic kernels on the same split operands, so
the results must agree bit for bit; each is also checked against the CPU oracle within the
tolerance the parity tests use. It also checks that the device's free memory does not move
across the second call. This file is collected last,
so a run that stops at the first failure has already run every other test.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from roofline_driven_tiling_gb300 import binding, inputs


def _tolerance(A: np.ndarray, B: np.ndarray) -> float:
    return 1e-6 * A.shape[1] * float(np.max(np.abs(A))) * float(np.max(np.abs(B)))


def test_noalloc_rejects_problems_beyond_the_scratch_array():
    import __graft_entry__
    __graft_entry__.build()
    f = binding.t2s_gemm_f32_tf32x3_noalloc
    fake = 1 << 20  # never dereferenced: the size check comes first
    # 8 * (4096 + 4096) * 4096 bytes of planes: far beyond 32 MiB.
    assert f(4096, 4096, 4096, fake, fake, fake + 4096) == binding.T2S_ERR_TOO_LARGE
    assert f(-1, 4, 4, fake, fake, fake + 4096) == binding.T2S_ERR_INVALID
    assert "32 MiB" in binding.t2s_status_string(binding.T2S_ERR_TOO_LARGE)
    size = binding.t2s_gemm_f32_tf32x3_workspace_size
    cap = binding.T2S_TF32X3_NOALLOC_MAX_SCRATCH
    # Four planes of 4-byte values, K padded to a multiple of 32: 1024^3 takes 16 MiB, and
    # 1440^3 is the largest square product that fits (1441 pads K to 1472).
    assert size(1024, 1024, 1024) == 16 << 20
    assert size(1440, 1440, 1440) <= cap < size(1441, 1441, 1441)
    assert f(1441, 1441, 1441, fake, fake, fake + 4096) == binding.T2S_ERR_TOO_LARGE


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream

    cases = [(1000, 1003, 997, 21), (384, 520, 200, 22)]  # second call: smaller, other K
    prepared = []
    for M, N, K, seed in cases:
        A = inputs.uniform(M, K, 100 + seed)
        B = inputs.uniform(K, N, 200 + seed)
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        C_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
        C_new = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        need = binding.t2s_gemm_f32_tf32x3_workspace_size(M, N, K)
        assert need <= binding.T2S_TF32X3_NOALLOC_MAX_SCRATCH
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        prepared.append((M, N, K, A, B, dA, dB, C_ref, C_new, ws, need))
    torch.cuda.synchronize()

    for call, (M, N, K, A, B, dA, dB, C_ref, C_new, ws, need) in enumerate(prepared):
        rc = binding.t2s_gemm_f32_tf32x3(M, N, K, dA.data_ptr(), dB.data_ptr(), C_ref.data_ptr(),
                                         ws.data_ptr(), need, stream)
        assert rc == binding.T2S_OK, binding.t2s_status_string(rc)
        free_before, _ = torch.cuda.mem_get_info()
        rc = binding.t2s_gemm_f32_tf32x3_noalloc(M, N, K, dA.data_ptr(), dB.data_ptr(),
                                                 C_new.data_ptr(), stream)
        assert rc == binding.T2S_OK, binding.t2s_status_string(rc)
        assert binding.t2s_device_status(stream) == binding.T2S_OK
        free_after, _ = torch.cuda.mem_get_info()
        if call > 0:
            # The scratch array was set up by the first call; later calls take no memory.
            assert free_after == free_before
        got = C_new.cpu().numpy()
        same_kernels = C_ref.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), same_kernels.view(np.uint32)), \
            "call %d differs from the workspace entry point" % call
        want = oracle.sgemm(A, B, oracle.MUL_ADD)
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - want))) <= _tolerance(A, B)
