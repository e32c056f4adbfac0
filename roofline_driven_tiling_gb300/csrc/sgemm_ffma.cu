// sgemm_ffma.cu -- the product kernel: FP32 C = A x B on the CUDA cores of sm_103a.
//
// What it computes is the definition on page "GEMM 커널 테스트 코드 작성 및 최적화
// (1024^3 크기 실험)", section "Naive GEMM 커널 동작 방식": one FP32 accumulator per C
// element, updated by a fused multiply-add for k = 0, 1, ..., K-1 in order. Zero
// padding beyond K appends fma(0, 0, acc) = acc steps, which change nothing, so the
// result is bit-identical to the definition evaluated with fmaf().
//
// How (page "4주차: Roofline과 Tiling", sections "3. Tiling" and item 8 of "이번 주차
// 핵심"): each CTA owns a BM x BN tile of C and walks K in BK-wide blocks. A and B
// blocks are staged in shared memory once and reused BN (resp. BM) times, which is
// what moves the kernel from the bandwidth slope to the FP32 compute roof.
//
// GB300 design:
//  * Warp specialisation. One producer warp fills a STAGES-deep ring of shared-memory
//    buffers; consumer warps compute. Each ring slot has a "full" mbarrier (data
//    landed) and an "empty" mbarrier (all consumer warps done reading it).
//  * Producer, aligned case (K % 4 == 0, N % 4 == 0, 16-byte aligned pointers): the
//    Tensor Memory Accelerator loads a BM x BK box of A and a BK x BN box of B per
//    stage; out-of-range elements of edge boxes are filled with zeros by the TMA
//    unit, and completion is counted in transaction bytes on the full barrier.
//  * Producer, general case: 4-byte cp.async copies with zero fill write the same
//    shared-memory image; each producer lane arrives on the full barrier when its
//    copies land (cp.async.mbarrier.arrive.noinc).
//  * A is stored K-major as it is in global memory (TMA cannot transpose 4-byte
//    elements). Rows of BK floats are XOR-swizzled in 16-byte chunks (the TMA
//    128/64/32-byte swizzle), so that the 8 rows a warp reads at one k chunk fall in
//    8 distinct bank groups. Each thread reads its A values as float4 along k.
//  * B is stored as it is (rows of BN floats); a warp reads 4 consecutive 16-byte
//    chunks of one row per load, which is conflict-free without a swizzle.
//  * Each consumer thread owns an 8 x 16 register tile of C: rows g + 8i of its
//    warp's 64 rows (g = lane / 4) and columns 4h + 16j + {0..3} of its warp's 64
//    columns (h = lane % 4). Accumulators are packed in pairs along n and updated
//    with fma.rn.f32x2: one instruction does two IEEE fused multiply-adds, which
//    halves the issue slots the FMAs need and leaves the rest for shared loads.
//  * Every barrier wait is bounded; on expiry the kernel records T2S_ERR_TIMEOUT in
//    the device status word and returns instead of hanging. The producer always
//    waits for its own in-flight copies before it exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "t2s_device.cuh"
#include "t2s_internal.h"
#include "t2s_tmap.h"

#ifndef BIG_AV
#define BIG_AV 2
#endif

namespace t2s {
namespace {

template <int BM_, int BN_, int BK_, int STAGES_, int WARPS_M_, int WARPS_N_, int MAX_REGS_,
          int AV_>
struct FfmaConfig {
  static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
  static constexpr int AV = AV_;  // k values per shared load of A (1, 2 or 4)
  static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
  static constexpr int MAX_REGS = MAX_REGS_;  // per thread; sets how many CTAs fit an SM
  static constexpr int TM = 8, TN = 16;  // per-thread C tile
  static constexpr int LM = 8, LN = 4;   // lanes along m and n (LM x LN = 32)
  static constexpr int WM = LM * TM, WN = LN * TN;
  static_assert(BM == WARPS_M * WM && BN == WARPS_N * WN, "tile / warp mismatch");
  static_assert(BK == 8 || BK == 16 || BK == 32, "A rows must be 32, 64 or 128 bytes");
  static_assert((AV == 1 || AV == 2 || AV == 4) && BK % AV == 0, "A load width");
  static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
  static constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
  static constexpr int A_ROW_BYTES = BK * 4;
  static constexpr int SWZ_MASK = A_ROW_BYTES / 16 - 1;  // 7 (128 B), 3 (64 B), 1 (32 B)
  static constexpr int A_STAGE_BYTES = BM * BK * 4;
  static constexpr int B_STAGE_BYTES = BK * BN * 4;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static_assert(A_STAGE_BYTES % 1024 == 0 && B_STAGE_BYTES % 1024 == 0, "stage alignment");
  // Ring buffers, 2 * STAGES barriers, and up to 1 KB to align the base to 1024 B
  // (the repeat of the 128-byte swizzle pattern).
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 2 * STAGES * 8 + 1024;
};

// Byte offset inside an A stage of 16-byte chunk `chunk` of row `row`, after the
// TMA swizzle: the chunk index is XORed with bits 7.. of the unswizzled offset.
template <class Cfg>
__device__ __forceinline__ uint32_t a_swizzled(uint32_t off) {
  return off ^ (((off >> 7) & Cfg::SWZ_MASK) << 4);
}

template <class Cfg, bool kTma>
__device__ __forceinline__ void producer(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                         const float* __restrict__ A, const float* __restrict__ B,
                                         int M, int N, int K, int m0, int n0, int nkb,
                                         uint32_t sA, uint32_t sB, uint32_t sBar, int lane,
                                         unsigned* status) {
  constexpr int S = Cfg::STAGES;
  auto full = [&](int s) { return sBar + 8u * s; };
  auto empty = [&](int s) { return sBar + 8u * (S + s); };
  int issued = 0;
  if (kTma) {
    if (lane == 0) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % S;
        const uint32_t round = static_cast<uint32_t>(kb / S);
        if (kb >= S && !mbar_wait_bounded(empty(s), (round - 1u) & 1u, status)) break;
        mbar_arrive_expect_tx(full(s), Cfg::STAGE_BYTES);
        tma_load_2d(sA + s * Cfg::A_STAGE_BYTES, tmA, kb * Cfg::BK, m0, full(s));
        tma_load_2d(sB + s * Cfg::B_STAGE_BYTES, tmB, n0, kb * Cfg::BK, full(s));
        issued = kb + 1;
      }
    }
  } else {
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % S;
      const uint32_t round = static_cast<uint32_t>(kb / S);
      if (kb >= S) {
        const bool freed = mbar_wait_bounded(empty(s), (round - 1u) & 1u, status);
        if (!__all_sync(0xffffffffu, freed)) break;
      }
      const int k0 = kb * Cfg::BK;
      const uint32_t a_dst = sA + s * Cfg::A_STAGE_BYTES;
#pragma unroll 4
      for (int e = lane; e < Cfg::BM * Cfg::BK; e += 32) {
        const int r = e / Cfg::BK, c = e % Cfg::BK;
        const int gm = m0 + r, gk = k0 + c;
        const bool v = gm < M && gk < K;
        const float* src = v ? A + (static_cast<int64_t>(gm) * K + gk) : A;
        cp_async_4(a_dst + a_swizzled<Cfg>(r * Cfg::A_ROW_BYTES + c * 4), src, v ? 4u : 0u);
      }
      const uint32_t b_dst = sB + s * Cfg::B_STAGE_BYTES;
#pragma unroll 4
      for (int e = lane; e < Cfg::BK * Cfg::BN; e += 32) {
        const int r = e / Cfg::BN, c = e % Cfg::BN;
        const int gk = k0 + r, gn = n0 + c;
        const bool v = gk < K && gn < N;
        const float* src = v ? B + (static_cast<int64_t>(gk) * N + gn) : B;
        cp_async_4(b_dst + (r * Cfg::BN + c) * 4, src, v ? 4u : 0u);
      }
      cp_async_arrive_noinc(full(s));
      issued = kb + 1;
    }
  }
  // Do not leave while copies into this CTA's shared memory are still in flight.
  if (kTma && lane != 0) return;
  const int first = issued > S ? issued - S : 0;
  for (int kb = first; kb < issued; ++kb) {
    if (!mbar_wait_bounded(full(kb % S), static_cast<uint32_t>(kb / S) & 1u, status)) break;
  }
}

template <class Cfg, bool kTma>
__global__ void __launch_bounds__(Cfg::THREADS) __maxnreg__(Cfg::MAX_REGS)
    sgemm_ffma_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const float* __restrict__ A,
                      const float* __restrict__ B, float* __restrict__ C, int M, int N, int K,
                      int tiles_m, int tiles_n, unsigned* status, int vec_store) {
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base;
  const uint32_t sB = sA + S * Cfg::A_STAGE_BYTES;
  const uint32_t sBar = sB + S * Cfg::B_STAGE_BYTES;

  // Grouped tile order: 8 tile-rows at a time sweep the columns, so that the A rows
  // and B columns in flight stay resident in L2.
  constexpr int kGroup = 8;
  const int tile = blockIdx.x;
  const int per_group = kGroup * tiles_n;
  const int first_m = (tile / per_group) * kGroup;
  const int gsz = min(tiles_m - first_m, kGroup);
  const int tm = first_m + (tile % per_group) % gsz;
  const int tn = (tile % per_group) / gsz;
  const int m0 = tm * Cfg::BM, n0 = tn * Cfg::BN;
  const int nkb = (K + Cfg::BK - 1) / Cfg::BK;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(sBar + 8u * s, kTma ? 1u : 32u);
      mbar_init(sBar + 8u * (S + s), Cfg::CONSUMER_WARPS);
    }
    mbar_fence_init();
  }
  if (kTma && warp == Cfg::CONSUMER_WARPS && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __syncthreads();

  if (warp == Cfg::CONSUMER_WARPS) {
    producer<Cfg, kTma>(&tmA, &tmB, A, B, M, N, K, m0, n0, nkb, sA, sB, sBar, lane, status);
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int wm0 = (warp % Cfg::WARPS_M) * Cfg::WM;
  const int wn0 = (warp / Cfg::WARPS_M) * Cfg::WN;
  const int g = lane >> 2, h = lane & 3;

  uint64_t acc[Cfg::TM][Cfg::TN / 2];
#pragma unroll
  for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
    for (int j = 0; j < Cfg::TN / 2; ++j) acc[i][j] = 0ull;  // two +0.0f

  // Row offsets (unswizzled) of this thread's 8 A rows, and the B column offset.
  const uint32_t a_row0 = static_cast<uint32_t>((wm0 + g) * Cfg::A_ROW_BYTES);
  const uint32_t b_col0 = static_cast<uint32_t>((wn0 + 4 * h) * 4);

  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb % S;
    // Every lane polls; the decision to give up is taken by the whole warp at once.
    const bool landed = mbar_wait_bounded(sBar + 8u * s, static_cast<uint32_t>(kb / S) & 1u, status);
    if (!__all_sync(0xffffffffu, landed)) return;
    const uint32_t a_base = sA + s * Cfg::A_STAGE_BYTES;
    const uint32_t b_base = sB + s * Cfg::B_STAGE_BYTES + b_col0;
#pragma unroll
    for (int kc = 0; kc < Cfg::BK / Cfg::AV; ++kc) {
      // AV consecutive k values of each of this thread's TM rows of A.
      float a[Cfg::TM][Cfg::AV];
#pragma unroll
      for (int i = 0; i < Cfg::TM; ++i)
        lds_vec<Cfg::AV>(a_base + a_swizzled<Cfg>(a_row0 + i * Cfg::LM * Cfg::A_ROW_BYTES +
                                                   kc * Cfg::AV * 4),
                         a[i]);
#pragma unroll
      for (int kk = 0; kk < Cfg::AV; ++kk) {
        uint64_t b[Cfg::TN / 2];
        const uint32_t b_row = b_base + (kc * Cfg::AV + kk) * (Cfg::BN * 4);
#pragma unroll
        for (int j = 0; j < Cfg::TN / 4; ++j) lds128_pairs(b_row + j * 64, b[2 * j], b[2 * j + 1]);
#pragma unroll
        for (int i = 0; i < Cfg::TM; ++i) {
          const uint64_t ap = pack_dup(a[i][kk]);
#pragma unroll
          for (int j = 0; j < Cfg::TN / 2; ++j) ffma2(acc[i][j], ap, b[j]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sBar + 8u * (S + s));
  }

  // ---------------------------------------------------------------- epilogue
  const int row0 = m0 + wm0 + g;
  const int col0 = n0 + wn0 + 4 * h;
#pragma unroll
  for (int i = 0; i < Cfg::TM; ++i) {
    const int row = row0 + i * Cfg::LM;
    if (row >= M) continue;
    float* crow = C + static_cast<int64_t>(row) * N;
#pragma unroll
    for (int j = 0; j < Cfg::TN / 4; ++j) {
      const int col = col0 + 16 * j;
      const float2 lo = unpack2(acc[i][2 * j]);
      const float2 hi = unpack2(acc[i][2 * j + 1]);
      if (vec_store) {
        if (col < N) *reinterpret_cast<float4*>(crow + col) = make_float4(lo.x, lo.y, hi.x, hi.y);
      } else {
        if (col + 0 < N) crow[col + 0] = lo.x;
        if (col + 1 < N) crow[col + 1] = lo.y;
        if (col + 2 < N) crow[col + 2] = hi.x;
        if (col + 3 < N) crow[col + 3] = hi.y;
      }
    }
  }
}

template <class Cfg, bool kTma>
cudaError_t run(const Problem& p) {
  CUtensorMap ta, tb;
  memset(&ta, 0, sizeof(ta));
  memset(&tb, 0, sizeof(tb));
  if (kTma) {
    const CUtensorMapSwizzle sw = Cfg::A_ROW_BYTES == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : Cfg::A_ROW_BYTES == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                           : CU_TENSOR_MAP_SWIZZLE_32B;
    cudaError_t e = encode_tmap_f32_2d(&ta, p.A, p.K, p.M, Cfg::BK, Cfg::BM, sw);
    if (e != cudaSuccess) return e;
    e = encode_tmap_f32_2d(&tb, p.B, p.N, p.K, Cfg::BN, Cfg::BK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  auto kern = sgemm_ffma_kernel<Cfg, kTma>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
  const int64_t tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
  const int64_t tiles = tiles_m * tiles_n;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int vec_store = (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) ? 1 : 0;
  kern<<<static_cast<unsigned>(tiles), Cfg::THREADS, Cfg::SMEM_BYTES, p.stream>>>(
      ta, tb, p.A, p.B, p.C, static_cast<int>(p.M), static_cast<int>(p.N), static_cast<int>(p.K),
      static_cast<int>(tiles_m), static_cast<int>(tiles_n), p.status, vec_store);
  return cudaGetLastError();
}

// 128 x 128 CTA tile, 4 consumer warps (2 x 2 of 64 x 64), BK = 32, 3 stages:
// 96 KB of ring per CTA, two CTAs per SM.
using Big = FfmaConfig<128, 128, 32, 3, 2, 2, 200, BIG_AV>;
// 64 x 128 tiles for products too small to give every SM two 128 x 128 tiles.
using Mid = FfmaConfig<64, 128, 32, 4, 1, 2, 200, 2>;
// 64 x 64 tiles, one consumer warp, for the smallest products.
using Small = FfmaConfig<64, 64, 32, 4, 1, 1, 200, 2>;

bool tma_ok(const Problem& p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p.A), b = reinterpret_cast<uintptr_t>(p.B);
  return p.K % 4 == 0 && p.N % 4 == 0 && (a & 15u) == 0 && (b & 15u) == 0;
}

template <class Cfg>
cudaError_t run_any(const Problem& p) {
  return tma_ok(p) ? run<Cfg, true>(p) : run<Cfg, false>(p);
}

}  // namespace

cudaError_t launch_ffma(const Problem& p) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t big_tiles = ((p.M + 127) / 128) * ((p.N + 127) / 128);
  const int64_t mid_tiles = ((p.M + 63) / 64) * ((p.N + 127) / 128);
  if (big_tiles >= 2 * static_cast<int64_t>(sms)) return run_any<Big>(p);
  if (mid_tiles >= static_cast<int64_t>(sms)) return run_any<Mid>(p);
  return run_any<Small>(p);
}

}  // namespace t2s
