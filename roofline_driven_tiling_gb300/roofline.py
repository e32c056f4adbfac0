"""Roofline model used to place measured GEMM points (reporting only).

The formulas follow page "4주차: Roofline과 Tiling":

* section "이번 주차 핵심", items 1-5, and section "1. Arithmetic Intensity":
  arithmetic intensity AI = FLOPs / bytes moved to and from HBM; attainable
  performance = min(peak FLOP/s, bandwidth x AI); the critical (ridge) AI is
  peak / bandwidth; below it a kernel is memory-bound, above it compute-bound.
* section "예시) Vector Add와 MatMul": vector add moves 12N bytes for N FLOPs
  (AI = 1/12); an N x N x N FP32 matmul moves 3N^2 x 4 bytes (read A and B,
  write C) for 2N^3 FLOPs (AI = N/6).

Page "GEMM 커널 테스트 코드 작성 및 최적화 (1024^3 크기 실험)", section
"수학적 정의", counts M*N*K multiplies plus M*N*K adds, i.e. 2MNK FLOPs, and
section "결과 해석" turns a time into GFLOP/s as FLOPs / seconds.

For an M x N x K product the byte count generalises the square case to
4 (MK + KN + MN): every element of A and B read once and every element of C
written once -- the algorithmic minimum, not what a kernel actually moves.

Peak figures for GB300 are not on the pages. The FP32 CUDA-core peak is built
from unit counts and clocks (SMs x FP32 lanes per SM x 2 FLOPs per FMA x clock);
memory and tensor peaks come from measurements passed in by the caller.
"""
from __future__ import annotations

FP32_BYTES = 4

#: GB300 unit counts used for the FP32 CUDA-core peak.
GB300_SMS = 152
FP32_LANES_PER_SM = 128
GB300_SM_MAX_MHZ = 2070.0


def gemm_flops(M: int, N: int, K: int) -> int:
    """FLOPs of C = A x B: M*N*K multiplies and M*N*K adds."""
    return 2 * int(M) * int(N) * int(K)


def gemm_bytes(M: int, N: int, K: int, elem_bytes: int = FP32_BYTES) -> int:
    """Algorithmic HBM bytes: read A (M x K) and B (K x N) once, write C (M x N) once."""
    return elem_bytes * (int(M) * int(K) + int(K) * int(N) + int(M) * int(N))


def vector_add_flops(n: int) -> int:
    """One add per element."""
    return int(n)


def vector_add_bytes(n: int, elem_bytes: int = FP32_BYTES) -> int:
    """Read two vectors and write one: 3 x n elements."""
    return 3 * elem_bytes * int(n)


def arithmetic_intensity(flops: float, nbytes: float) -> float:
    """FLOPs per byte moved to or from HBM."""
    if nbytes <= 0:
        raise ValueError("byte count must be positive")
    return float(flops) / float(nbytes)


def gemm_ai(M: int, N: int, K: int) -> float:
    return arithmetic_intensity(gemm_flops(M, N, K), gemm_bytes(M, N, K))


def attainable(peak_flops: float, bandwidth: float, ai: float) -> float:
    """Roofline ceiling min(peak, bandwidth x AI), in the units of peak_flops."""
    return min(float(peak_flops), float(bandwidth) * float(ai))


def ridge_ai(peak_flops: float, bandwidth: float) -> float:
    """Critical AI where the bandwidth slope meets the compute roof."""
    return float(peak_flops) / float(bandwidth)


def bound(ai: float, peak_flops: float, bandwidth: float) -> str:
    """'memory' below the ridge point, 'compute' at or above it."""
    return "memory" if ai < ridge_ai(peak_flops, bandwidth) else "compute"


def gflops(flops: float, seconds: float) -> float:
    """Achieved GFLOP/s for a kernel that ran `flops` in `seconds`."""
    return float(flops) / float(seconds) / 1e9


def fp32_peak_tflops(sms: int = GB300_SMS, mhz: float = GB300_SM_MAX_MHZ,
                     lanes: int = FP32_LANES_PER_SM) -> float:
    """FP32 CUDA-core peak: SMs x lanes x 2 FLOPs per FMA x clock, in TFLOP/s."""
    return sms * lanes * 2.0 * mhz * 1e6 / 1e12


#: FP64 fused multiply-adds per SM per clock on GB300: NVIDIA's nominal 1.25 TFLOP/s FP64 for
#: the whole GPU is 152 SMs x 2 FMA x 2 FLOP x 2.07 GHz = 1.26 TFLOP/s.
FP64_FMA_PER_SM_CLK = 2
FP64_PEAK_BASIS = "152 SMs x 2 FP64 FMA/clk x 2 FLOP x 2070 MHz (nominal 1.25 TFLOP/s)"


def fp64_peak_tflops(sms: int = GB300_SMS, mhz: float = GB300_SM_MAX_MHZ,
                     fma_per_clk: int = FP64_FMA_PER_SM_CLK) -> float:
    """FP64 CUDA-core peak: SMs x FP64 FMAs per clock x 2 FLOPs x clock, in TFLOP/s."""
    return sms * fma_per_clk * 2.0 * mhz * 1e6 / 1e12


def place(flops: float, seconds: float, nbytes: float, peak_tflops: float,
          bw_gbs: float) -> dict:
    """Place one measured point on the roofline.

    Returns the achieved TFLOP/s, the AI (with `nbytes`, algorithmic or measured),
    the ceiling min(peak, BW x AI) at that AI, the fraction of that ceiling, and
    whether the point sits left or right of the ridge.
    """
    achieved = flops / seconds / 1e12
    ai = arithmetic_intensity(flops, nbytes)
    roof = attainable(peak_tflops, bw_gbs / 1e3, ai)  # GB/s x FLOP/B -> TFLOP/s
    return {
        "tflops": achieved,
        "ai": ai,
        "roof_tflops": roof,
        "frac_of_roof": achieved / roof,
        "ridge_ai": ridge_ai(peak_tflops, bw_gbs / 1e3),
        "region": bound(ai, peak_tflops, bw_gbs / 1e3),
    }
