"""The C ABI without a GPU: the library loads, exports what the header declares,
and rejects bad arguments before touching CUDA."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from roofline_driven_tiling_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "t2s_gemm.h")


def header_functions():
    with open(HEADER, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(t2s_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return binding.lib()


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("t2s_gemm_f32", "t2s_gemm_f32_naive", "t2s_gemm_f32_smem32",
                     "t2s_gemm_f32_tf32x3", "t2s_gemm_f32_tf32x3_workspace_size",
                     "t2s_status_string", "t2s_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), "libt2s_gemm.so does not export %s" % name
        assert name in binding.SIGNATURES, "binding lacks %s" % name


def test_binding_declares_nothing_the_header_lacks():
    assert set(binding.SIGNATURES) == set(header_functions())


def test_status_strings(lib):
    for code in range(0, 6):
        s = binding.t2s_status_string(code)
        assert isinstance(s, str) and s
    assert binding.t2s_status_string(binding.T2S_OK) == "ok"


@pytest.mark.parametrize("fn", ["t2s_gemm_f32", "t2s_gemm_f32_naive", "t2s_gemm_f32_smem32"])
def test_invalid_arguments_rejected_on_host(lib, fn):
    f = getattr(binding, fn)
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    assert f(-1, 4, 4, fake, fake, fake + 4096) == binding.T2S_ERR_INVALID
    assert f(4, -1, 4, fake, fake, fake + 4096) == binding.T2S_ERR_INVALID
    assert f(4, 4, -1, fake, fake, fake + 4096) == binding.T2S_ERR_INVALID
    big = binding.T2S_MAX_DIM + 1
    assert f(big, 4, 4, fake, fake, fake + 4096) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, 0, fake, fake + 4096) == binding.T2S_ERR_INVALID  # NULL A
    assert f(4, 4, 4, fake, 0, fake + 4096) == binding.T2S_ERR_INVALID  # NULL B
    assert f(4, 4, 4, fake, fake, 0) == binding.T2S_ERR_INVALID  # NULL C
    assert f(4, 4, 4, fake + 2, fake, fake + 4096) == binding.T2S_ERR_INVALID  # misaligned
    assert f(4, 4, 4, fake, fake, fake) == binding.T2S_ERR_INVALID  # C aliases A
    assert f(4, 4, 4, fake + 4096, fake, fake) == binding.T2S_ERR_INVALID  # C aliases B


@pytest.mark.parametrize("fn", ["t2s_gemm_f32", "t2s_gemm_f32_naive", "t2s_gemm_f32_smem32"])
def test_empty_output_is_a_noop(lib, fn):
    f = getattr(binding, fn)
    # M == 0 or N == 0: nothing to compute; NULL is fine for empty matrices.
    assert f(0, 0, 0, 0, 0, 0) == binding.T2S_OK
    assert f(0, 7, 0, 0, 0, 0) == binding.T2S_OK
    assert f(5, 0, 0, 0, 0, 0) == binding.T2S_OK


def test_tf32x3_workspace_size(lib):
    ws = binding.t2s_gemm_f32_tf32x3_workspace_size
    # Two planes (big, small) of A (M x K) and of B (N x K), 4 bytes each, 256-byte padded.
    assert ws(4096, 4096, 4096) == 4 * 4 * 4096 * 4096
    # K is padded to a multiple of 32 in the planes.
    assert ws(128, 128, 997) == 4 * 4 * 128 * 1024
    assert ws(0, 0, 0) == 0
    assert ws(-1, 2, 3) == 0
    assert ws(3, 5, 7) % 256 == 0 and ws(3, 5, 7) >= 2 * 4 * (3 * 7 + 5 * 7)
    fake = 1 << 20
    assert binding.t2s_gemm_f32_tf32x3(-1, 4, 4, fake, fake, fake + 4096, fake, 1 << 20) == \
        binding.T2S_ERR_INVALID


def test_version(lib):
    assert binding.t2s_version() >= 100


def test_host_pipeline_rejects_bad_arguments(lib):
    f = binding.t2s_gemm_f32_host
    fake = 1 << 20
    ok = dict(hA=fake, hB=fake + 4096, hC=fake + 8192, dA=fake + 12288, dB=fake + 16384,
              dC=fake + 20480)
    def call(M, N, K, **kw):
        a = dict(ok, **kw)
        return f(M, N, K, a["hA"], a["hB"], a["hC"], a["dA"], a["dB"], a["dC"], 0)
    assert call(-1, 4, 4) == binding.T2S_ERR_INVALID
    assert call(4, 4, binding.T2S_MAX_DIM + 1) == binding.T2S_ERR_INVALID
    for name in ok:
        assert call(4, 4, 4, **{name: 0}) == binding.T2S_ERR_INVALID, name
    assert call(4, 4, 4, dC=ok["dA"]) == binding.T2S_ERR_INVALID
    assert call(0, 4, 4) == binding.T2S_OK  # nothing to do


def test_vector_add_rejects_bad_arguments(lib):
    f = binding.t2s_vector_add_f32
    fake = 1 << 20
    assert f(-1, fake, fake + 64, fake + 128) == binding.T2S_ERR_INVALID
    assert f(8, 0, fake + 64, fake + 128) == binding.T2S_ERR_INVALID
    assert f(8, fake + 2, fake + 64, fake + 128) == binding.T2S_ERR_INVALID
    assert f(8, fake, fake + 64, fake) == binding.T2S_ERR_INVALID  # z aliases x
    assert f(0, 0, 0, 0) == binding.T2S_OK


def test_splitk_workspace_size_and_arguments(lib):
    ws = binding.t2s_gemm_f32_splitk_workspace_size
    assert ws(1024, 512, 4096, 4) == 4 * 1024 * 512 * 4
    assert ws(1024, 512, 4096, 1) == 0  # one chunk: no partial planes
    assert ws(16, 16, 40, 8) == 2 * 16 * 16 * 4  # chunks round up to 32 values: 2 planes
    assert ws(16, 16, 40, 65) == 0 and ws(-1, 2, 3, 2) == 0
    fake = 1 << 20
    assert binding.t2s_gemm_f32_splitk(4, 4, 4, fake, fake + 64, fake + 128, 65, fake, 1 << 20, 0) == \
        binding.T2S_ERR_INVALID
    assert binding.t2s_gemm_f32_splitk(-1, 4, 4, fake, fake + 64, fake + 128, 2, fake, 1 << 20, 0) == \
        binding.T2S_ERR_INVALID


def test_bf16_workspace_size_and_arguments(lib):
    ws = binding.t2s_gemm_bf16_f32_workspace_size
    # B transposed (N x Kp) and a padded A plane (M x Kp), 2 bytes each, Kp = K rounded up to
    # 64, each plane 256-byte padded.
    assert ws(4096, 4096, 4096) == 2 * 2 * 4096 * 4096
    assert ws(128, 64, 997) == 2 * 128 * 1024 + 2 * 64 * 1024
    assert ws(0, 0, 0) == 0 and ws(-1, 2, 3) == 0
    assert ws(3, 5, 7) % 256 == 0
    fake = 1 << 20
    f = binding.t2s_gemm_bf16_f32
    assert f(-1, 4, 4, fake, fake + 64, fake + 4096, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake + 1, fake + 64, fake + 4096, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake, fake + 64, fake + 4098, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake, fake + 64, fake, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(0, 4, 4, 0, fake + 64, 0, 0, 0, 0) == binding.T2S_OK  # M = 0: nothing to do


@pytest.mark.parametrize("fn", ["t2s_gemm_f64", "t2s_gemm_f64_naive", "t2s_gemm_f64_smem32"])
def test_f64_entries_reject_bad_arguments(lib, fn):
    f = getattr(binding, fn)
    fake = 1 << 20
    assert f(-1, 4, 4, fake, fake + 256, fake + 512, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake + 4, fake + 256, fake + 512, 0) == binding.T2S_ERR_INVALID  # 4-aligned
    assert f(4, 4, 4, fake, fake + 256, fake + 516, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake, fake + 256, fake, 0) == binding.T2S_ERR_INVALID  # C == A
    assert f(4, 4, 4, 0, fake + 256, fake + 512, 0) == binding.T2S_ERR_INVALID  # NULL A
    assert f(0, 4, 4, 0, fake + 256, 0, 0) == binding.T2S_OK  # M = 0: nothing to do


def test_f16_entry_matches_bf16_contract(lib):
    for M, N, K in [(4096, 4096, 4096), (128, 64, 997), (3, 5, 7), (0, 0, 0)]:
        assert binding.t2s_gemm_f16_f32_workspace_size(M, N, K) == \
            binding.t2s_gemm_bf16_f32_workspace_size(M, N, K)
    fake = 1 << 20
    f = binding.t2s_gemm_f16_f32
    assert f(-1, 4, 4, fake, fake + 64, fake + 4096, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake + 1, fake + 64, fake + 4096, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake, fake + 64, fake, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(0, 4, 4, 0, fake + 64, 0, 0, 0, 0) == binding.T2S_OK


def test_streamk_arguments(lib):
    assert binding.t2s_gemm_f32_streamk_workspace_size(-1, 4, 4) == 0
    fake = 1 << 20
    f = binding.t2s_gemm_f32_streamk
    assert f(-1, 4, 4, fake, fake + 64, fake + 128, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(4, 4, 4, fake, fake + 64, fake, fake, 1 << 20, 0) == binding.T2S_ERR_INVALID
    assert f(0, 4, 4, 0, fake + 64, 0, 0, 0, 0) == binding.T2S_OK


def test_probes_reject_bad_arguments(lib):
    """The throughput probes check their arguments before touching a device."""
    import ctypes
    flops = ctypes.c_int64(0)
    fake = 1 << 20  # never dereferenced: the checks come first
    fp = ctypes.addressof(flops)
    assert lib.t2s_probe_fp32_fma(0, fake, fp, 0) == binding.T2S_ERR_INVALID
    assert lib.t2s_probe_fp32_fma((1 << 24) + 1, fake, fp, 0) == binding.T2S_ERR_INVALID
    assert lib.t2s_probe_fp32_fma(10, None, fp, 0) == binding.T2S_ERR_INVALID
    assert lib.t2s_probe_fp32_fma(10, fake, None, 0) == binding.T2S_ERR_INVALID
    assert lib.t2s_probe_tf32_mma(0, fake, fp, 0) == binding.T2S_ERR_INVALID
    assert lib.t2s_probe_tf32_mma((1 << 16) + 1, fake, fp, 0) == binding.T2S_ERR_INVALID
    assert lib.t2s_probe_tf32_mma(10, None, fp, 0) == binding.T2S_ERR_INVALID
    # The store probe: whole 256 x 128 tiles, a 16-byte aligned C, mode 0 or 1.
    st = lib.t2s_probe_store_f32
    for args in [(0, 128, fake, 0), (255, 128, fake, 0), (256, 127, fake, 0), (512, 100, fake, 1),
                 (256, 128, None, 0), (256, 128, fake + 4, 0), (256, 128, fake, 2),
                 (256, 128, fake, -1), ((1 << 30) + 256, 128, fake, 0)]:
        assert st(*args, 1.0, fp, 0) == binding.T2S_ERR_INVALID, args
    assert st(256, 128, fake, 0, 1.0, None, 0) == binding.T2S_ERR_INVALID
