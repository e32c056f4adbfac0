"""The roofline model against the figures the pages print."""
from __future__ import annotations

import math

import pytest

from golden_io import page_figures
from roofline_driven_tiling_gb300 import roofline as rl


def test_flops_of_1024_cubed():
    fig = page_figures()
    assert rl.gemm_flops(1024, 1024, 1024) == 2 * 1024 ** 3
    assert rl.gemm_flops(1024, 1024, 1024) == pytest.approx(fig["flops_1024_cubed"], rel=1e-3)


@pytest.mark.parametrize("ms_key,gf_key", [("naive_ms_1024", "naive_gflops_1024"),
                                           ("tiled_ms_1024", "tiled_gflops_1024")])
def test_gflops_from_page_times(ms_key, gf_key):
    fig = page_figures()
    g = rl.gflops(rl.gemm_flops(1024, 1024, 1024), fig[ms_key] / 1e3)
    assert round(g) == pytest.approx(fig[gf_key], abs=1.0)


def test_time_ratio():
    fig = page_figures()
    assert fig["tiled_ms_1024"] / fig["naive_ms_1024"] == pytest.approx(fig["tiled_over_naive"], abs=1e-4)


def test_vector_add_ai():
    fig = page_figures()
    n = 1 << 20
    ai = rl.arithmetic_intensity(rl.vector_add_flops(n), rl.vector_add_bytes(n))
    assert ai == pytest.approx(1.0 / 12.0)
    assert round(ai, 3) == fig["ai_vector_add"]


def test_square_matmul_ai():
    fig = page_figures()
    assert rl.gemm_bytes(256, 256, 256) == fig["matmul_bytes_per_n2"] * 256 ** 2
    assert rl.gemm_ai(256, 256, 256) == pytest.approx(256 / 6)
    assert round(rl.gemm_ai(256, 256, 256), 2) == fig["ai_matmul_n256"]
    for n in (1, 7, 128, 4096):
        assert rl.gemm_ai(n, n, n) == pytest.approx(n / 6)


def test_rectangular_ai_reduces_to_square():
    # The general M, N, K form equals N/6 for squares and is symmetric in M and N.
    assert rl.gemm_ai(1000, 1003, 997) == pytest.approx(rl.gemm_ai(1003, 1000, 997))
    assert rl.gemm_ai(16384, 16384, 32) == pytest.approx(2 * 16384 * 16384 * 32 /
                                                         (4 * (2 * 16384 * 32 + 16384 ** 2)))


def test_roofline_min_and_ridge():
    peak, bw = 80.0, 8.0  # TFLOP/s, TB/s
    assert rl.ridge_ai(peak, bw) == 10.0
    assert rl.attainable(peak, bw, 2.0) == 16.0  # bandwidth slope
    assert rl.attainable(peak, bw, 100.0) == peak  # compute roof
    assert rl.bound(9.99, peak, bw) == "memory"
    assert rl.bound(10.0, peak, bw) == "compute"
    # The slope is continuous at the ridge.
    assert rl.attainable(peak, bw, rl.ridge_ai(peak, bw)) == pytest.approx(peak)


def test_fp32_peak_from_units():
    # 152 SMs x 128 lanes x 2 FLOPs x 2.07 GHz
    assert rl.fp32_peak_tflops() == pytest.approx(152 * 128 * 2 * 2.07e9 / 1e12)
    assert rl.fp32_peak_tflops(mhz=1000.0, sms=1, lanes=1) == pytest.approx(2e-3)


def test_place_point():
    p = rl.place(flops=2 * 4096 ** 3, seconds=2e-3, nbytes=rl.gemm_bytes(4096, 4096, 4096),
                 peak_tflops=80.0, bw_gbs=8000.0)
    assert p["tflops"] == pytest.approx(2 * 4096 ** 3 / 2e-3 / 1e12)
    assert p["region"] == "compute"
    assert p["roof_tflops"] == 80.0
    assert math.isclose(p["frac_of_roof"], p["tflops"] / 80.0)
    low = rl.place(flops=1e9, seconds=1e-3, nbytes=1e9, peak_tflops=80.0, bw_gbs=8000.0)
    assert low["region"] == "memory" and low["roof_tflops"] == pytest.approx(8.0)


def test_sweep_covers_the_sweep_configuration():
    """The roofline sweep tool measures the square shapes 128^3 .. 8192^3, the two low-AI
    shapes and the ragged one, for every FP32 entry point (no GPU needed to check this)."""
    from roofline_driven_tiling_gb300 import sweep
    squares = {(n, n, n) for n in (128, 256, 512, 1024, 2048, 4096, 8192)}
    assert squares <= set(sweep.SHAPES)
    assert {(16384, 16384, 32), (8192, 8192, 64), (1000, 1003, 997)} <= set(sweep.SHAPES)
    # Every FP32 entry point, and the vendor library's product as a comparison column.
    assert set(sweep.KERNELS) == {"ffma", "tf32x3", "splitk", "streamk", "smem32", "naive", "cublas"}
