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
//  * A STAGES-deep ring of shared-memory buffers per CTA, one "full" mbarrier per slot.
//    On the TMA path there is no producer warp: every warp computes. CTA tiles run from
//    32 x 32 to 256 x 128 of 4 or 8 warps, chosen per shape (pick_ffma), and an SM holds at
//    least 8 warps, two per sub-partition (16 for the small register tiles), at up to 255
//    registers per thread for the largest register tile.
//  * Aligned case (K % 4 == 0, N % 4 == 0, 16-byte aligned pointers): the Tensor Memory
//    Accelerator loads a BM x BK box of A and a BK x BN box of B per stage; elements
//    outside the matrices are filled with zeros by the TMA unit, and completion is
//    counted in transaction bytes on the full barrier. The last warp to finish reading a
//    slot (a shared-memory counter per slot) issues the refill, so no warp ever blocks
//    waiting for another to free a slot.
//  * General case (K or N not a multiple of 4, or A or B not 16-byte aligned: row strides
//    TMA cannot take): stages are copied with 4-byte cp.async and zero fill into the same
//    shared-memory image, a whole A row per warp instruction, and a copying thread arrives
//    on the full barrier when its copies land (cp.async.mbarrier.arrive.noinc); an "empty"
//    barrier per slot counts the warps done with it. The 8-warp tiles, which run one CTA
//    per SM, add 4 producer warps that make every copy up to 6 stages ahead
//    (sgemm_ffma_general_ws_kernel); the others copy with every thread, each warp
//    refilling the slot of the previous K block after its current one
//    (sgemm_ffma_general_kernel).
//  * Short K (at most 3 K blocks, at least two rounds of 256 x 128 tiles): a persistent grid
//    whose warps hand C to TMA stores while the ring loads the next tile
//    (sgemm_ffma_pstore_kernel).
//  * A is stored K-major as it is in global memory (TMA cannot transpose 4-byte
//    elements). Rows of BK floats (of 32 in each 32-deep sub-block when BK = 64) are
//    XOR-swizzled in 16-byte chunks (the TMA 128/64/32-byte swizzle), so that the 8 rows a
//    warp reads at one k chunk fall in 8 distinct bank groups.
//  * B is stored as it is (rows of BN floats); a warp reads 4 consecutive 16-byte
//    chunks of one row per load, which is conflict-free without a swizzle.
//  * Each thread owns a TM x TN register tile of C (8 x 16 in the large CTA tiles; 8 x 8,
//    8 x 4, 7 x 4 or 4 x 8 in the small ones): rows g + 8i of its warp's 8 TM rows
//    (g = lane / 4) and columns 4h + 16j + {0..3} of its warp's 4 TN columns (h = lane % 4).
//    Accumulators are packed in pairs along n and updated with fma.rn.f32x2: one
//    instruction does two IEEE fused multiply-adds, which halves the issue slots the
//    FMAs need and leaves the rest for shared loads.
//  * The k loop runs in groups of 8 k values (fully unrolled inside a group) so that the
//    loop body stays small enough for the instruction cache; the large tiles unroll the
//    whole K block when K is long enough to pay for the code, and the small ones load the
//    fragments of step k + 1 while step k is multiplied.
//  * Every barrier wait is bounded; on expiry the kernel records T2S_ERR_TIMEOUT in the
//    device status word and returns instead of hanging, after letting its own in-flight
//    copies land.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "t2s_device.cuh"
#include "t2s_internal.h"
#include "t2s_tmap.h"

namespace t2s {
namespace {

template <int BM_, int BN_, int BK_, int STAGES_, int WARPS_M_, int WARPS_N_, int AV_, int TM_,
          int TN_, int KG_UNROLL_>
struct FfmaConfig {
  static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_;
  static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
  static constexpr int AV = AV_;          // k values per shared load of A (1, 2 or 4)
  static constexpr int TM = TM_, TN = TN_;  // per-thread C tile
  static constexpr int KG_UNROLL = KG_UNROLL_;  // groups of 8 k unrolled together
  static constexpr int LM = 8, LN = 4;    // lanes along m and n (LM x LN = 32)
  static constexpr int WM = LM * TM, WN = LN * TN;
  static_assert(BM == WARPS_M * WM && BN == WARPS_N * WN, "tile / warp mismatch");
  static_assert(TN % 4 == 0 && TM >= 1, "columns come in float4 chunks");
  static_assert(BK == 8 || BK == 16 || BK == 32 || BK == 64, "A rows of 32, 64 or 128 bytes");
  static_assert((AV == 1 || AV == 2 || AV == 4) && 8 % AV == 0, "A load width");
  static constexpr int WARPS = WARPS_M * WARPS_N;
  static constexpr int THREADS = WARPS * 32;
  // Warps per SM the register file should hold: two per SM sub-partition for the
  // 128-accumulator tile (up to 255 registers), more for smaller tiles.
  static constexpr int TARGET_WARPS = TM * TN >= 128 ? 8 : TM * TN >= 64 ? 12 : 16;
  static constexpr int MIN_BLOCKS = TARGET_WARPS / WARPS > 0 ? TARGET_WARPS / WARPS : 1;
  // A is staged as BK / BKS sub-blocks of BKS k values (BK = 64: two of 32), each BM rows of
  // BKS floats in the TMA swizzle, one after the other.
  static constexpr int BKS = BK > 32 ? 32 : BK;
  static constexpr int A_SUBS = BK / BKS;
  static constexpr int A_ROW_BYTES = BKS * 4;
  static constexpr int A_SUB_BYTES = BM * BKS * 4;
  static constexpr int SWZ_MASK = A_ROW_BYTES / 16 - 1;  // 7 (128 B), 3 (64 B), 1 (32 B)
  static constexpr int A_STAGE_BYTES = BM * BK * 4;
  static constexpr int B_STAGE_BYTES = BK * BN * 4;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static_assert(A_STAGE_BYTES % 1024 == 0 && B_STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(A_SUB_BYTES % 1024 == 0, "sub-block alignment (the swizzle's 1 KB repeat)");
  // Ring, full[S] and empty[S] barriers, refill counters, and up to 1 KB to align the
  // base to 1024 B (the repeat of the 128-byte swizzle pattern).
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 2 * STAGES * 8 + STAGES * 4 + 1024;
};

// Byte offset inside an A stage after the TMA swizzle: the 16-byte chunk index is XORed
// with bits 7.. of the unswizzled offset.
template <class Cfg>
__device__ __forceinline__ uint32_t a_swizzled(uint32_t off) {
  return off ^ (((off >> 7) & Cfg::SWZ_MASK) << 4);
}

// Ring depth of the general (cp.async) path: one stage more than the TMA path where the
// extra stage still fits the CTAs per SM the configuration is built for. The general path
// issues a stage's copies S - 2 K blocks before it is needed (see sgemm_ffma_general_kernel),
// so the extra stage is what hides the copies' latency.
template <class Cfg>
struct GenRing {
  static constexpr int ringBytes(int s) { return s * Cfg::STAGE_BYTES + 2 * s * 8 + 1024; }
  // 228 KB of shared memory per SM, 1 KB of it reserved per CTA.
  static constexpr bool kDeeper = Cfg::MIN_BLOCKS * (ringBytes(Cfg::STAGES + 1) + 1024) <= 228 * 1024;
  static constexpr int STAGES = kDeeper ? Cfg::STAGES + 1 : Cfg::STAGES;
  static constexpr int SMEM_BYTES = ringBytes(STAGES);
};

// One stage of the general path: the BM x BK block of A at (m0, k0) and the BK x BN block of B
// at (k0, n0), copied with 4-byte cp.async by the NT threads of a copy group (t = 0 .. NT - 1:
// every thread of the CTA, or its producer warps) into the same shared-memory image the TMA
// path writes (A K-major with the 128-byte swizzle, B as stored), zeros for rows >= M,
// k >= kend and columns >= N. Warp w of the group copies the A rows w, w + NT / 32, ... (lane =
// k, one instruction per row and 32-deep sub-block); the group copies B rows NT / BN at a time
// (thread t: column t % BN). A stage wholly inside the matrices takes no bounds checks. The thread arrives on the
// stage's full barrier once its copies have landed.
template <class Cfg, int NT>
__device__ __forceinline__ void gen_copy_stage(const float* __restrict__ A,
                                               const float* __restrict__ B, int M, int N, int K,
                                               int kend, int m0, int n0, int k0, uint32_t a_dst,
                                               uint32_t b_dst, uint32_t full_bar, int t) {
  constexpr int NW = NT / 32;
  static_assert(Cfg::BKS == 32, "one warp instruction per A row and sub-block");
  static_assert(NT % 32 == 0 && Cfg::BM % NW == 0 && NT % Cfg::BN == 0, "copy mapping");
  constexpr int A_ROWS = Cfg::BM / NW;   // A rows per warp
  constexpr int B_STEP = NT / Cfg::BN;   // B rows per pass of the group
  constexpr int B_PASSES = Cfg::BK / B_STEP;
  const int warp = t >> 5, lane = t & 31;
  const int bcol = t % Cfg::BN, brow = t / Cfg::BN;
  // This thread's first A element (row `warp`, k = k0 + lane) and first B element (row
  // k0 + brow, column n0 + bcol).
  const float* a_src = A + static_cast<int64_t>(m0 + warp) * K + (k0 + lane);
  const float* b_src = B + static_cast<int64_t>(k0 + brow) * N + (n0 + bcol);
  const uint32_t b_dst0 = b_dst + static_cast<uint32_t>((brow * Cfg::BN + bcol) * 4);
  auto a_off = [&](int r) {  // swizzled offset of (row r, k = lane) in the A stage
    return static_cast<uint32_t>(r * Cfg::A_ROW_BYTES +
                                 ((((lane >> 2) ^ (r & 7)) << 4) | ((lane & 3) << 2)));
  };
  if (m0 + Cfg::BM <= M && k0 + Cfg::BK <= kend && n0 + Cfg::BN <= N) {
#pragma unroll
    for (int sb = 0; sb < Cfg::A_SUBS; ++sb)
#pragma unroll
      for (int i = 0; i < A_ROWS; ++i) {
        const int r = warp + NW * i;
        cp_async_4_full(a_dst + sb * Cfg::A_SUB_BYTES + a_off(r),
                        a_src + sb * 32 + static_cast<int64_t>(NW) * i * K);
      }
#pragma unroll
    for (int i = 0; i < B_PASSES; ++i)
      cp_async_4_full(b_dst0 + static_cast<uint32_t>(i * B_STEP * Cfg::BN * 4),
                      b_src + static_cast<int64_t>(B_STEP) * i * N);
  } else {
    // Out-of-range elements are zero-filled; their source pointer is replaced by the
    // matrix's first element, which nothing reads (0 source bytes).
    const int rows_left = M - m0 - warp;
#pragma unroll
    for (int sb = 0; sb < Cfg::A_SUBS; ++sb) {
      const bool k_ok = k0 + sb * 32 + lane < kend;
#pragma unroll
      for (int i = 0; i < A_ROWS; ++i) {
        const int r = warp + NW * i;
        const bool v = k_ok && NW * i < rows_left;
        cp_async_4(a_dst + sb * Cfg::A_SUB_BYTES + a_off(r),
                   v ? a_src + sb * 32 + static_cast<int64_t>(NW) * i * K : A, v ? 4u : 0u);
      }
    }
    const bool n_ok = n0 + bcol < N;
    const int k_left = kend - k0 - brow;
#pragma unroll
    for (int i = 0; i < B_PASSES; ++i) {
      const bool v = n_ok && B_STEP * i < k_left;
      cp_async_4(b_dst0 + static_cast<uint32_t>(i * B_STEP * Cfg::BN * 4),
                 v ? b_src + static_cast<int64_t>(B_STEP) * i * N : B, v ? 4u : 0u);
    }
  }
  cp_async_arrive_noinc(full_bar);
}

// The general path with producer warps, for the 8-warp tiles that run one CTA per SM and
// leave registers for 4 more warps: the producers make every copy, S stages ahead, and the
// compute warps only wait for stages to land. Ring depth: the most stages up to 6 that fit.
constexpr int kProducerThreads = 128;
template <class Cfg>
struct WsRing {
  static constexpr int ringBytes(int s) { return s * Cfg::STAGE_BYTES + 2 * s * 8 + 1024; }
  static constexpr int STAGES = ringBytes(6) <= 200 * 1024   ? 6
                                : ringBytes(5) <= 200 * 1024 ? 5
                                : ringBytes(4) <= 200 * 1024 ? 4
                                                             : 3;
  static constexpr int SMEM_BYTES = ringBytes(STAGES);
  static constexpr int THREADS = Cfg::THREADS + kProducerThreads;
  // The compute warps' registers (tiles of at most 64 accumulators per thread) plus the
  // producers' must fit one CTA per SM.
  static constexpr bool kUsable = Cfg::WARPS == 8 && Cfg::TM * Cfg::TN <= 64;
};

// One TMA stage: a BM x BK box of A and a BK x BN box of B, completion counted in bytes.
template <class Cfg>
__device__ __forceinline__ void tma_stage(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                          int m0, int n0, int k0, uint32_t a_dst,
                                          uint32_t b_dst, uint32_t full_bar) {
  mbar_arrive_expect_tx(full_bar, Cfg::STAGE_BYTES);
#pragma unroll
  for (int sb = 0; sb < Cfg::A_SUBS; ++sb)
    tma_load_2d(a_dst + sb * Cfg::A_SUB_BYTES, tmA, k0 + sb * Cfg::BKS, m0, full_bar);
  tma_load_2d(b_dst, tmB, n0, k0, full_bar);
}

// One K block of the register-tile product: groups of 8 k values of A and B fragments from
// the stage at a_base (this thread's first A row) and b_base (its first B column), fused
// multiply-adds into acc in ascending k.
template <class Cfg>
__device__ __forceinline__ void ffma_kblock_direct(uint64_t (&acc)[Cfg::TM][Cfg::TN / 2],
                                                   uint32_t a_base, uint32_t b_base,
                                                   uint32_t xr) {
#pragma unroll Cfg::KG_UNROLL
  for (int kg = 0; kg < Cfg::BK / 8; ++kg) {
    // 8 k values = two 16-byte chunks of each A row of sub-block kg / (BKS / 8), swizzled.
    constexpr int KGS = Cfg::BKS / 8;
    const uint32_t kgl = static_cast<uint32_t>(kg % KGS);
    const uint32_t sub = static_cast<uint32_t>(kg / KGS) * Cfg::A_SUB_BYTES;
    const uint32_t c0 = sub + (((2u * kgl) ^ xr) << 4), c1 = sub + (((2u * kgl + 1u) ^ xr) << 4);
    const uint32_t b_kg = b_base + kg * (8 * Cfg::BN * 4);
#pragma unroll
    for (int kv = 0; kv < 8 / Cfg::AV; ++kv) {
      const uint32_t koff = (kv * Cfg::AV < 4 ? c0 : c1) + (kv * Cfg::AV % 4) * 4;
      float a[Cfg::TM][Cfg::AV];
#pragma unroll
      for (int i = 0; i < Cfg::TM; ++i)
        lds_vec<Cfg::AV>(a_base + i * Cfg::LM * Cfg::A_ROW_BYTES + koff, a[i]);
#pragma unroll
      for (int kk = 0; kk < Cfg::AV; ++kk) {
        uint64_t b[Cfg::TN / 2];
        const uint32_t b_row = b_kg + (kv * Cfg::AV + kk) * (Cfg::BN * 4);
#pragma unroll
        for (int j = 0; j < Cfg::TN / 4; ++j) lds128_pairs(b_row + j * 64, b[2 * j], b[2 * j + 1]);
        // Column pairs outer, rows inner: consecutive FMAs share the B pair. Measured 3 %
        // faster than rows outer at 4096^3 and 8192^3 (hoisting the {a, a} moves alone
        // changes nothing, so the gain is in operand reuse, not in the moves); 2 x 2 blocks of
        // (row, column pair) measured the same as this order.
        uint64_t ap[Cfg::TM];
#pragma unroll
        for (int i = 0; i < Cfg::TM; ++i) ap[i] = pack_dup(a[i][kk]);
#pragma unroll
        for (int j = 0; j < Cfg::TN / 2; ++j)
#pragma unroll
          for (int i = 0; i < Cfg::TM; ++i) ffma2(acc[i][j], ap[i], b[j]);
      }
    }
  }
}

// The same K block with the fragments of k step k + 1 loaded while step k is multiplied (two
// register sets). It pays where few warps share a sub-partition and latency shows: tiles of at
// most 64 accumulators per thread (1024^3 with 128 x 64 tiles: 37.0 -> 39.9 TFLOP/s; 2048^3
// with 64 x 64 tiles: 52.3 -> 54.0). It made the 128-accumulator tile slower (4096^3: 62.9 ->
// 61.2; B alone one step ahead: 60.8), which keeps the direct form.
template <class Cfg>
__device__ __forceinline__ void ffma_kblock_pipelined(uint64_t (&acc)[Cfg::TM][Cfg::TN / 2],
                                                      uint32_t a_base, uint32_t b_base,
                                                      uint32_t xr) {
  // A in groups of AV k values (one load per row every AV steps), B per step; each loaded one
  // step (A: one group) ahead into the other register set.
  constexpr int AV = Cfg::AV;
  float a[2][Cfg::TM][AV];
  uint64_t b[2][Cfg::TN / 2];
  auto load_a = [&](int kq, int buf) {
    const int kql = kq % Cfg::BKS;
    const uint32_t koff = static_cast<uint32_t>(kq / Cfg::BKS) * Cfg::A_SUB_BYTES +
                          ((static_cast<uint32_t>(kql >> 2) ^ xr) << 4) + (kql & 3) * 4;
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
      lds_vec<AV>(a_base + i * Cfg::LM * Cfg::A_ROW_BYTES + koff, a[buf][i]);
  };
  auto load_b = [&](int k, int buf) {
    const uint32_t b_row = b_base + k * (Cfg::BN * 4);
#pragma unroll
    for (int j = 0; j < Cfg::TN / 4; ++j)
      lds128_pairs(b_row + j * 64, b[buf][2 * j], b[buf][2 * j + 1]);
  };
  load_a(0, 0);
  load_b(0, 0);
#pragma unroll
  for (int k = 0; k < Cfg::BK; ++k) {
    const int cur = k & 1, abuf = (k / AV) & 1;
    if (k + 1 < Cfg::BK) load_b(k + 1, cur ^ 1);
    if (k % AV == 0 && k + AV < Cfg::BK) load_a(k + AV, abuf ^ 1);
    uint64_t ap[Cfg::TM];
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i) ap[i] = pack_dup(a[abuf][i][k % AV]);
#pragma unroll
    for (int j = 0; j < Cfg::TN / 2; ++j)
#pragma unroll
      for (int i = 0; i < Cfg::TM; ++i) ffma2(acc[i][j], ap[i], b[cur][j]);
  }
}

template <class Cfg>
__device__ __forceinline__ void ffma_kblock(uint64_t (&acc)[Cfg::TM][Cfg::TN / 2], uint32_t a_base,
                                            uint32_t b_base, uint32_t xr) {
  if constexpr (Cfg::TM * Cfg::TN <= 64) {
    ffma_kblock_pipelined<Cfg>(acc, a_base, b_base, xr);
  } else {
    ffma_kblock_direct<Cfg>(acc, a_base, b_base, xr);
  }
}

// Stores this thread's C tile (rows row0 + 8i, column chunks col0 + 16j) into the row-major
// matrix C of M x N (ld = N), skipping what lies outside it.
template <class Cfg>
__device__ __forceinline__ void store_tile(const uint64_t (&acc)[Cfg::TM][Cfg::TN / 2], float* C,
                                           int M, int N, int row0, int col0, int vec_store) {
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

__device__ __forceinline__ uint64_t pack_pair(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// Loads this thread's C tile (the positions store_tile writes) into the accumulators; +0.0f
// outside C.
template <class Cfg>
__device__ __forceinline__ void load_tile(uint64_t (&acc)[Cfg::TM][Cfg::TN / 2], const float* C,
                                          int M, int N, int row0, int col0, int vec_load) {
#pragma unroll
  for (int i = 0; i < Cfg::TM; ++i) {
    const int row = row0 + i * Cfg::LM;
    const float* crow = C + static_cast<int64_t>(row < M ? row : 0) * N;
#pragma unroll
    for (int j = 0; j < Cfg::TN / 4; ++j) {
      const int col = col0 + 16 * j;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < M) {
        if (vec_load) {
          if (col < N) v = *reinterpret_cast<const float4*>(crow + col);
        } else {
          if (col + 0 < N) v.x = crow[col + 0];
          if (col + 1 < N) v.y = crow[col + 1];
          if (col + 2 < N) v.z = crow[col + 2];
          if (col + 3 < N) v.w = crow[col + 3];
        }
      }
      acc[i][2 * j] = pack_pair(v.x, v.y);
      acc[i][2 * j + 1] = pack_pair(v.z, v.w);
    }
  }
}

// The CTA's tile and K range. Grouped tile order over the tiles_m x tiles_n grid of wbm x wbn
// tiles: 8 tile-rows at a time sweep the columns, so that the A rows and B columns in flight
// stay resident in L2. A launch covers tiles tile_off, tile_off + 1, ... of that order, each as
// dm x dn CTA tiles of BM x BN (wbm = dm BM, wbn = dn BN); CTA tiles wholly outside C have no
// work (returns false). The K range is chunk blockIdx.y of k_chunk values from k_base on (the
// whole of K when the grid has one row and k_base is 0), written to plane blockIdx.y of C;
// k_chunk and k_base are multiples of BK.
template <class Cfg>
__device__ __forceinline__ bool cta_work(int M, int N, int K, int tiles_m, int tiles_n, int wbm,
                                         int wbn, int tile_off, int dm, int dn, int k_chunk,
                                         int k_base, int& m0, int& n0, int& kbeg, int& kend) {
  constexpr int kGroup = 8;
  const int tile = tile_off + static_cast<int>(blockIdx.x) / (dm * dn);
  const int sub = static_cast<int>(blockIdx.x) % (dm * dn);
  const int per_group = kGroup * tiles_n;
  const int first_m = (tile / per_group) * kGroup;
  const int gsz = min(tiles_m - first_m, kGroup);
  m0 = (first_m + (tile % per_group) % gsz) * wbm + (sub / dn) * Cfg::BM;
  n0 = ((tile % per_group) / gsz) * wbn + (sub % dn) * Cfg::BN;
  kbeg = k_base + static_cast<int>(blockIdx.y) * k_chunk;
  kend = min(K, kbeg + k_chunk);
  return m0 < M && n0 < N;
}

// The product on the TMA path (K % 4 == 0, N % 4 == 0, 16-byte aligned A and B).
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS)
    sgemm_ffma_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const float* __restrict__ A,
                      const float* __restrict__ B, float* __restrict__ C, int M, int N, int K,
                      int tiles_m, int tiles_n, unsigned* status, int vec_store, int k_chunk,
                      int64_t c_plane, int wbm, int wbn, int tile_off, int dm, int dn,
                      int k_base, int accumulate) {
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base;
  const uint32_t sB = sA + S * Cfg::A_STAGE_BYTES;
  const uint32_t sBar = sB + S * Cfg::B_STAGE_BYTES;  // full[S] (the empty[S] words are unused)
  const uint32_t sCnt = sBar + 16u * S;                // refill counters
  auto full = [&](int s) { return sBar + 8u * s; };
  auto a_stage = [&](int s) { return sA + static_cast<uint32_t>(s) * Cfg::A_STAGE_BYTES; };
  auto b_stage = [&](int s) { return sB + static_cast<uint32_t>(s) * Cfg::B_STAGE_BYTES; };

  int m0, n0, kbeg, kend;
  if (!cta_work<Cfg>(M, N, K, tiles_m, tiles_n, wbm, wbn, tile_off, dm, dn, k_chunk, k_base, m0,
                     n0, kbeg, kend))
    return;
  C += static_cast<int64_t>(blockIdx.y) * c_plane;
  const int nkb = (kend - kbeg + Cfg::BK - 1) / Cfg::BK;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1u);
      asm volatile("st.shared.u32 [%0], 0;" ::"r"(sCnt + 4u * s) : "memory");
    }
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int kb = 0; kb < S && kb < nkb; ++kb)
      tma_stage<Cfg>(&tmA, &tmB, m0, n0, kbeg + kb * Cfg::BK, a_stage(kb), b_stage(kb), full(kb));
  }
  __syncthreads();

  const int wm0 = (warp % Cfg::WARPS_M) * Cfg::WM;
  const int wn0 = (warp / Cfg::WARPS_M) * Cfg::WN;
  const int g = lane >> 2, h = lane & 3;

  uint64_t acc[Cfg::TM][Cfg::TN / 2];
  if (accumulate) {
    // Continue the sums already in C (the product over the K values before kbeg): each
    // accumulator resumes from the FP32 value it was stored as, so the chain of fused
    // multiply-adds is the same as in one pass over all of K.
    load_tile<Cfg>(acc, C, M, N, m0 + wm0 + g, n0 + wn0 + 4 * h, vec_store);
  } else {
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
      for (int j = 0; j < Cfg::TN / 2; ++j) acc[i][j] = 0ull;  // two +0.0f
  }

  // This thread's A rows are wm0 + g + 8i: every one has the same swizzle XOR (the row
  // index mod 8 is g), so the swizzle reduces to XORing the chunk index with `xr`.
  const uint32_t a_row0 = static_cast<uint32_t>((wm0 + g) * Cfg::A_ROW_BYTES);
  const uint32_t xr = (a_row0 >> 7) & Cfg::SWZ_MASK;
  const uint32_t b_col0 = static_cast<uint32_t>((wn0 + 4 * h) * 4);

  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb % S;
    // Every lane polls; the decision to give up is taken by the whole warp at once.
    const bool landed = mbar_wait_bounded(full(s), static_cast<uint32_t>(kb / S) & 1u, status);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) {
        // Let copies already issued into this CTA's ring land before leaving.
        for (int j = kb; j < kb + S && j < nkb; ++j)
          mbar_wait_bounded(full(j % S), static_cast<uint32_t>(j / S) & 1u, status, 10000000ull);
      }
      return;
    }
    ffma_kblock<Cfg>(acc, a_stage(s) + a_row0, b_stage(s) + b_col0, xr);
    __syncwarp();
    if (lane == 0) {
      // The last warp to finish with this slot refills it with stage kb + S.
      if (slot_done_count(sCnt + 4u * s) == Cfg::WARPS - 1) {
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(sCnt + 4u * s) : "memory");
        if (kb + S < nkb)
          tma_stage<Cfg>(&tmA, &tmB, m0, n0, kbeg + (kb + S) * Cfg::BK, a_stage(s), b_stage(s),
                         full(s));
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  store_tile<Cfg>(acc, C, M, N, m0 + wm0 + g, n0 + wn0 + 4 * h, vec_store);
}

// The product on the general path (any K and N, 4-byte aligned A and B): the same register
// tiles and k order as the TMA path, over a ring of GenRing<Cfg>::STAGES slots that every
// thread fills with gen_copy_stage. Per K block kb, a warp waits for stage kb to land (a full
// barrier counting every thread's copies), multiplies it, and marks the slot done (an empty
// barrier counting warps). Only then does it wait for every warp to be done with stage
// kb - 1 and copy its share of stage kb - 1 + S into that slot: a warp may run a K block ahead
// of the slowest one without waiting, and each stage is issued S - 2 K blocks before it is
// used.
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS)
    sgemm_ffma_general_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB, const float* __restrict__ A,
                              const float* __restrict__ B, float* __restrict__ C, int M, int N,
                              int K, int tiles_m, int tiles_n, unsigned* status, int vec_store,
                              int k_chunk, int64_t c_plane, int wbm, int wbn, int tile_off, int dm,
                              int dn, int k_base, int accumulate) {
  (void)tmA;
  (void)tmB;
  constexpr int S = GenRing<Cfg>::STAGES;
  static_assert(S >= 3, "a stage is issued S - 2 K blocks ahead");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base;
  const uint32_t sB = sA + S * Cfg::A_STAGE_BYTES;
  const uint32_t sBar = sB + S * Cfg::B_STAGE_BYTES;  // full[S], empty[S]
  auto full = [&](int s) { return sBar + 8u * s; };
  auto empty = [&](int s) { return sBar + 8u * (S + s); };
  auto a_stage = [&](int s) { return sA + static_cast<uint32_t>(s) * Cfg::A_STAGE_BYTES; };
  auto b_stage = [&](int s) { return sB + static_cast<uint32_t>(s) * Cfg::B_STAGE_BYTES; };

  int m0, n0, kbeg, kend;
  if (!cta_work<Cfg>(M, N, K, tiles_m, tiles_n, wbm, wbn, tile_off, dm, dn, k_chunk, k_base, m0,
                     n0, kbeg, kend))
    return;
  C += static_cast<int64_t>(blockIdx.y) * c_plane;
  const int nkb = (kend - kbeg + Cfg::BK - 1) / Cfg::BK;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), static_cast<uint32_t>(Cfg::THREADS));
      mbar_init(empty(s), static_cast<uint32_t>(Cfg::WARPS));
    }
    mbar_fence_init();
  }
  __syncthreads();
  // Prologue: stages 0 .. S - 2 (slot S - 1 is filled after the first K block).
  for (int kb = 0; kb < S - 1 && kb < nkb; ++kb)
    gen_copy_stage<Cfg, Cfg::THREADS>(A, B, M, N, K, kend, m0, n0, kbeg + kb * Cfg::BK,
                                      a_stage(kb), b_stage(kb), full(kb),
                                      static_cast<int>(threadIdx.x));

  const int wm0 = (warp % Cfg::WARPS_M) * Cfg::WM;
  const int wn0 = (warp / Cfg::WARPS_M) * Cfg::WN;
  const int g = lane >> 2, h = lane & 3;

  uint64_t acc[Cfg::TM][Cfg::TN / 2];
  if (accumulate) {
    load_tile<Cfg>(acc, C, M, N, m0 + wm0 + g, n0 + wn0 + 4 * h, vec_store);
  } else {
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
      for (int j = 0; j < Cfg::TN / 2; ++j) acc[i][j] = 0ull;  // two +0.0f
  }

  const uint32_t a_row0 = static_cast<uint32_t>((wm0 + g) * Cfg::A_ROW_BYTES);
  const uint32_t xr = (a_row0 >> 7) & Cfg::SWZ_MASK;
  const uint32_t b_col0 = static_cast<uint32_t>((wn0 + 4 * h) * 4);

  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb % S;
    // Every lane polls; the decision to give up is taken by the whole warp at once. A thread
    // that gives up first waits for its own copies to land, so none lands after it exits.
    const bool landed = mbar_wait_bounded(full(s), static_cast<uint32_t>(kb / S) & 1u, status);
    if (!__all_sync(0xffffffffu, landed)) {
      asm volatile("cp.async.wait_all;" ::: "memory");
      return;
    }
    ffma_kblock<Cfg>(acc, a_stage(s) + a_row0, b_stage(s) + b_col0, xr);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
    // Refill: stage kb + S - 1 goes into the slot of stage kb - 1 once every warp is done
    // with that (the slot S - 1 is still free after the first K block).
    const int nk = kb + S - 1;
    if (nk < nkb) {
      const int ns = nk % S;
      bool freed = true;
      if (kb >= 1) freed = mbar_wait_bounded(empty(ns), static_cast<uint32_t>((kb - 1) / S) & 1u, status);
      if (!__all_sync(0xffffffffu, freed)) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        return;
      }
      gen_copy_stage<Cfg, Cfg::THREADS>(A, B, M, N, K, kend, m0, n0, kbeg + nk * Cfg::BK,
                                        a_stage(ns), b_stage(ns), full(ns),
                                        static_cast<int>(threadIdx.x));
    }
  }

  // ---------------------------------------------------------------- epilogue
  store_tile<Cfg>(acc, C, M, N, m0 + wm0 + g, n0 + wn0 + 4 * h, vec_store);
}

// The general path with producer warps (WsRing<Cfg>::kUsable configurations): warps
// 0 .. WARPS - 1 compute as in the TMA kernel; warps WARPS .. WARPS + 3 copy stage j into ring
// slot j % S once every compute warp is done with stage j - S (an empty barrier counting compute
// warps), then arrive on the slot's full barrier (counting producer threads) when their copies
// land. A compute warp never waits for another, only for its stages to land.
template <class Cfg>
__global__ void __launch_bounds__(WsRing<Cfg>::THREADS, 1)
    sgemm_ffma_general_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                                 const __grid_constant__ CUtensorMap tmB,
                                 const float* __restrict__ A, const float* __restrict__ B,
                                 float* __restrict__ C, int M, int N, int K, int tiles_m,
                                 int tiles_n, unsigned* status, int vec_store, int k_chunk,
                                 int64_t c_plane, int wbm, int wbn, int tile_off, int dm, int dn,
                                 int k_base, int accumulate) {
  (void)tmA;
  (void)tmB;
  constexpr int S = WsRing<Cfg>::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base;
  const uint32_t sB = sA + S * Cfg::A_STAGE_BYTES;
  const uint32_t sBar = sB + S * Cfg::B_STAGE_BYTES;  // full[S], empty[S]
  auto full = [&](int s) { return sBar + 8u * s; };
  auto empty = [&](int s) { return sBar + 8u * (S + s); };
  auto a_stage = [&](int s) { return sA + static_cast<uint32_t>(s) * Cfg::A_STAGE_BYTES; };
  auto b_stage = [&](int s) { return sB + static_cast<uint32_t>(s) * Cfg::B_STAGE_BYTES; };

  int m0, n0, kbeg, kend;
  if (!cta_work<Cfg>(M, N, K, tiles_m, tiles_n, wbm, wbn, tile_off, dm, dn, k_chunk, k_base, m0,
                     n0, kbeg, kend))
    return;
  C += static_cast<int64_t>(blockIdx.y) * c_plane;
  const int nkb = (kend - kbeg + Cfg::BK - 1) / Cfg::BK;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), static_cast<uint32_t>(kProducerThreads));
      mbar_init(empty(s), static_cast<uint32_t>(Cfg::WARPS));
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp >= Cfg::WARPS) {
    // ------------------------------------------------ producers
    const int t = static_cast<int>(threadIdx.x) - Cfg::THREADS;
    for (int j = 0; j < nkb; ++j) {
      const int s = j % S;
      if (j >= S) {
        const bool freed = mbar_wait_bounded(empty(s), static_cast<uint32_t>((j - S) / S) & 1u, status);
        if (!__all_sync(0xffffffffu, freed)) break;
      }
      gen_copy_stage<Cfg, kProducerThreads>(A, B, M, N, K, kend, m0, n0, kbeg + j * Cfg::BK,
                                            a_stage(s), b_stage(s), full(s), t);
    }
    // None of this thread's copies lands after it exits.
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // ------------------------------------------------ compute warps
  const int wm0 = (warp % Cfg::WARPS_M) * Cfg::WM;
  const int wn0 = (warp / Cfg::WARPS_M) * Cfg::WN;
  const int g = lane >> 2, h = lane & 3;

  uint64_t acc[Cfg::TM][Cfg::TN / 2];
  if (accumulate) {
    load_tile<Cfg>(acc, C, M, N, m0 + wm0 + g, n0 + wn0 + 4 * h, vec_store);
  } else {
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
      for (int j = 0; j < Cfg::TN / 2; ++j) acc[i][j] = 0ull;  // two +0.0f
  }
  const uint32_t a_row0 = static_cast<uint32_t>((wm0 + g) * Cfg::A_ROW_BYTES);
  const uint32_t xr = (a_row0 >> 7) & Cfg::SWZ_MASK;
  const uint32_t b_col0 = static_cast<uint32_t>((wn0 + 4 * h) * 4);

  for (int kb = 0; kb < nkb; ++kb) {
    const int s = kb % S;
    const bool landed = mbar_wait_bounded(full(s), static_cast<uint32_t>(kb / S) & 1u, status);
    if (!__all_sync(0xffffffffu, landed)) return;  // compute warps issue no copies
    ffma_kblock<Cfg>(acc, a_stage(s) + a_row0, b_stage(s) + b_col0, xr);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
  }

  // ---------------------------------------------------------------- epilogue
  store_tile<Cfg>(acc, C, M, N, m0 + wm0 + g, n0 + wn0 + 4 * h, vec_store);
}

// Persistent product with a TMA-store epilogue, for short K, where storing C takes about as
// long as the multiply-adds (a 16384 x 16384 C is 1 GB): one CTA per SM walks tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... of the grouped order, and its TMA ring of S stages
// runs on across tiles (iteration j of the CTA is K block j % nkb of its tile j / nkb, so the
// last warp to finish with a slot refills it with iteration j + S). Each warp multiplies its
// 64 x 64 part of a tile exactly as the product kernel does (one CTA per tile, k ascending: the
// same bits), then copies its sums into its own 16 KB of shared memory (two 64-row x 32-column
// boxes, 128-byte swizzle) and hands them to the TMA unit, which stores them while the warp
// goes on to the next tile. Before reusing the boxes a warp waits until its previous stores
// have read them; before exiting, until they are complete.
// PASSES: the warp stores its 64 x 64 part in that many passes of 64 / PASSES rows (two boxes
// of 64 / PASSES rows x 32 columns each), so that its staging holds one pass; between passes
// the warp waits until the previous pass's stores have read the boxes.
template <class Cfg, int S, int PASSES>
struct PStore {
  static_assert(Cfg::WM == 64 && Cfg::WN == 64, "64 x 64 warp tiles: two 32-column boxes each");
  static_assert(PASSES == 1 || PASSES == 2, "whole 8-row groups per pass");
  static constexpr int ROWS = 64 / PASSES;
  static constexpr int BOX_BYTES = ROWS * 128;
  static constexpr int STAGING_BYTES = Cfg::WARPS * 2 * BOX_BYTES;
  static constexpr int SMEM_BYTES =
      S * Cfg::STAGE_BYTES + STAGING_BYTES + 2 * S * 8 + S * 4 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
};

template <class Cfg, int S, int PASSES>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS)
    sgemm_ffma_pstore_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, int M, int N, int K,
                             int tiles_m, int tiles_n, unsigned* status) {
  using P = PStore<Cfg, S, PASSES>;
  (void)M;
  (void)N;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base;
  const uint32_t sB = sA + S * Cfg::A_STAGE_BYTES;
  const uint32_t sStg = sB + S * Cfg::B_STAGE_BYTES;  // 1024-byte aligned (stage sizes are)
  const uint32_t sBar = sStg + P::STAGING_BYTES;      // full[S], then refill counters
  const uint32_t sCnt = sBar + 16u * S;
  auto full = [&](int s) { return sBar + 8u * s; };
  auto a_stage = [&](int s) { return sA + static_cast<uint32_t>(s) * Cfg::A_STAGE_BYTES; };
  auto b_stage = [&](int s) { return sB + static_cast<uint32_t>(s) * Cfg::B_STAGE_BYTES; };
  auto origin = [&](int tile, int& m0, int& n0) {
    constexpr int kGroup = 8;
    const int per_group = kGroup * tiles_n;
    const int first_m = (tile / per_group) * kGroup;
    const int gsz = min(tiles_m - first_m, kGroup);
    m0 = (first_m + (tile % per_group) % gsz) * Cfg::BM;
    n0 = ((tile % per_group) / gsz) * Cfg::BN;
  };
  const int tiles = tiles_m * tiles_n;
  const int nkb = (K + Cfg::BK - 1) / Cfg::BK;
  const int my_tiles = (tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);
  const int64_t iters = static_cast<int64_t>(my_tiles) * nkb;
  // Loads iteration q of this CTA into ring slot s.
  auto issue = [&](int64_t q, int s) {
    int m0, n0;
    origin(static_cast<int>(blockIdx.x + (q / nkb) * gridDim.x), m0, n0);
    tma_stage<Cfg>(&tmA, &tmB, m0, n0, static_cast<int>(q % nkb) * Cfg::BK, a_stage(s),
                   b_stage(s), full(s));
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1u);
      asm volatile("st.shared.u32 [%0], 0;" ::"r"(sCnt + 4u * s) : "memory");
    }
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    for (int s = 0; s < S && s < iters; ++s) issue(s, s);
  }
  __syncthreads();

  const int wm0 = (warp % Cfg::WARPS_M) * Cfg::WM;
  const int wn0 = (warp / Cfg::WARPS_M) * Cfg::WN;
  const int g = lane >> 2, h = lane & 3;
  const uint32_t a_row0 = static_cast<uint32_t>((wm0 + g) * Cfg::A_ROW_BYTES);
  const uint32_t xr = (a_row0 >> 7) & Cfg::SWZ_MASK;
  const uint32_t b_col0 = static_cast<uint32_t>((wn0 + 4 * h) * 4);
  const uint32_t stg = sStg + static_cast<uint32_t>(warp) * 2u * P::BOX_BYTES;
  int64_t j = 0;  // iterations consumed
  for (int t = 0; t < my_tiles; ++t) {
    uint64_t acc[Cfg::TM][Cfg::TN / 2];
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
      for (int q = 0; q < Cfg::TN / 2; ++q) acc[i][q] = 0ull;  // two +0.0f
    for (int kb = 0; kb < nkb; ++kb, ++j) {
      const int s = static_cast<int>(j % S);
      const bool landed = mbar_wait_bounded(full(s), static_cast<uint32_t>(j / S) & 1u, status);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) {
          // Let copies already issued into this CTA's ring land, and this warp's stores
          // complete, before leaving.
          for (int64_t q = j; q < j + S && q < iters; ++q)
            mbar_wait_bounded(full(static_cast<int>(q % S)), static_cast<uint32_t>(q / S) & 1u,
                              status, 10000000ull);
          bulk_wait_all();
        }
        return;
      }
      ffma_kblock<Cfg>(acc, a_stage(s) + a_row0, b_stage(s) + b_col0, xr);
      __syncwarp();
      if (lane == 0 && slot_done_count(sCnt + 4u * s) == Cfg::WARPS - 1) {
        // The last warp to finish with this slot refills it with iteration j + S.
        asm volatile("st.shared.u32 [%0], 0;" ::"r"(sCnt + 4u * s) : "memory");
        if (j + S < iters) issue(j + S, s);
      }
    }
    // Epilogue, pass by pass: once this warp's previous stores have read its boxes, rows
    // g + 8i of the pass and column chunk h + 4q of its 64 x 64 part go to box q / 2, 16-byte
    // chunk (h + 4 (q % 2)) ^ g of row g + 8i within the pass (the 128-byte swizzle). A
    // 16-byte store is served a quarter-warp (lanes of g = 2t, 2t + 1) at a time, and those two
    // rows' swizzles differ in bit 0 only, so at step q lanes of odd g store chunk q ^ 1 of the
    // box instead of q: the eight lanes then fill the eight 16-byte bank groups once each.
    int m0, n0;
    origin(static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x), m0, n0);
#pragma unroll
    for (int pass = 0; pass < PASSES; ++pass) {
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
#pragma unroll
      for (int ii = 0; ii < Cfg::TM / PASSES; ++ii) {
        const int i = pass * (Cfg::TM / PASSES) + ii;
        const uint32_t row = static_cast<uint32_t>(g + 8 * ii) * 128u;
#pragma unroll
        for (int q = 0; q < Cfg::TN / 4; ++q) {
          const bool odd = (g & 1) != 0;
          const int qq = q ^ 1;  // the other chunk of the same box
          const uint64_t v0 = odd ? acc[i][2 * qq] : acc[i][2 * q];
          const uint64_t v1 = odd ? acc[i][2 * qq + 1] : acc[i][2 * q + 1];
          const int qs = odd ? qq : q;
          const uint32_t chunk = static_cast<uint32_t>((h + 4 * (qs % 2)) ^ g);
          const float2 lo = unpack2(v0), hi = unpack2(v1);
          st_shared_v4(stg + static_cast<uint32_t>(q / 2) * P::BOX_BYTES + row + (chunk << 4),
                       __float_as_uint(lo.x), __float_as_uint(lo.y), __float_as_uint(hi.x),
                       __float_as_uint(hi.y));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // The TMA unit clips the boxes at the edges of C.
        const int y = m0 + wm0 + pass * P::ROWS;
        tma_store_2d(&tmC, stg, n0 + wn0, y);
        tma_store_2d(&tmC, stg + P::BOX_BYTES, n0 + wn0 + 32, y);
      }
    }
  }
  // Every store has completed before the CTA's shared memory goes away.
  if (lane == 0) bulk_wait_all();
}

// A run of the grouped tile order: tiles [off, off + count) of C cut into wbm x wbn tiles
// (count < 0: to the end). Zero sizes stand for the configuration's own tile.
struct TilePart {
  int wbm = 0, wbn = 0;
  int64_t off = 0, count = -1;
  // K values [k0, k0 + kc) only (kc > 0, multiples of 32), added onto the values in C when
  // `accumulate` is set.
  int64_t k0 = 0, kc = 0;
  int accumulate = 0;
};

// Launches the kernel over `splits` K chunks of k_chunk values each (splits == 1: the whole
// product into p.C). Chunk z writes plane z of `out`, planes M x N apart. `part` limits the
// launch to a run of tiles, each computed as CTA tiles of the configuration.
template <class Cfg, bool kTma>
cudaError_t run(const Problem& p, int splits = 1, int k_chunk = 0, float* out = nullptr,
                TilePart part = TilePart()) {
  CUtensorMap ta, tb;
  memset(&ta, 0, sizeof(ta));
  memset(&tb, 0, sizeof(tb));
  if (kTma) {
    const CUtensorMapSwizzle sw = Cfg::A_ROW_BYTES == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : Cfg::A_ROW_BYTES == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                           : CU_TENSOR_MAP_SWIZZLE_32B;
    cudaError_t e = encode_tmap_f32_2d(&ta, p.A, p.K, p.M, Cfg::BKS, Cfg::BM, sw);
    if (e != cudaSuccess) return e;
    e = encode_tmap_f32_2d(&tb, p.B, p.N, p.K, Cfg::BN, Cfg::BK, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  // The kernel of this path; only the ones a configuration can run are instantiated.
  using Kernel = void (*)(const CUtensorMap, const CUtensorMap, const float*, const float*, float*,
                          int, int, int, int, int, unsigned*, int, int, int64_t, int, int, int,
                          int, int, int, int);
  Kernel kern;
  int smem, threads;
  if constexpr (kTma) {
    kern = sgemm_ffma_kernel<Cfg>;
    smem = Cfg::SMEM_BYTES;
    threads = Cfg::THREADS;
  } else if constexpr (WsRing<Cfg>::kUsable) {
    kern = sgemm_ffma_general_ws_kernel<Cfg>;
    smem = WsRing<Cfg>::SMEM_BYTES;
    threads = WsRing<Cfg>::THREADS;
  } else {
    kern = sgemm_ffma_general_kernel<Cfg>;
    smem = GenRing<Cfg>::SMEM_BYTES;
    threads = Cfg::THREADS;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int wbm = part.wbm > 0 ? part.wbm : Cfg::BM, wbn = part.wbn > 0 ? part.wbn : Cfg::BN;
  if (wbm % Cfg::BM != 0 || wbn % Cfg::BN != 0) return cudaErrorInvalidConfiguration;
  const int dm = wbm / Cfg::BM, dn = wbn / Cfg::BN;
  const int64_t tiles_m = (p.M + wbm - 1) / wbm;
  const int64_t tiles_n = (p.N + wbn - 1) / wbn;
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t count = part.count < 0 ? tiles - part.off : part.count;
  if (part.off < 0 || count < 0 || part.off + count > tiles) return cudaErrorInvalidConfiguration;
  if (count == 0) return cudaSuccess;
  if (count * dm * dn > 0x7fffffffLL || splits < 1 || splits > 65535)
    return cudaErrorInvalidConfiguration;
  float* c = out != nullptr ? out : p.C;
  const int vec_store = (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(c) & 15u) == 0) ? 1 : 0;
  if (part.kc > 0 && (splits != 1 || part.k0 % 32 != 0 || part.kc % 32 != 0 || part.k0 < 0 ||
                      part.k0 >= p.K))
    return cudaErrorInvalidConfiguration;
  const int chunk = part.kc > 0 ? static_cast<int>(part.kc)
                    : splits == 1 ? static_cast<int>(p.K) : k_chunk;
  const dim3 grid(static_cast<unsigned>(count * dm * dn), static_cast<unsigned>(splits));
  kern<<<grid, threads, smem, p.stream>>>(
      ta, tb, p.A, p.B, c, static_cast<int>(p.M), static_cast<int>(p.N), static_cast<int>(p.K),
      static_cast<int>(tiles_m), static_cast<int>(tiles_n), p.status, vec_store, chunk,
      p.M * p.N, wbm, wbn, static_cast<int>(part.off), dm, dn, static_cast<int>(part.k0),
      part.accumulate);
  return cudaGetLastError();
}

// 128 x 128 CTA tile, 4 warps (2 x 2 of 64 x 64), 8 x 16 per thread, BK = 32, 3 stages:
// 96 KB of ring per CTA, two CTAs (8 warps) per SM. The k loop is fully unrolled over a K
// block when K is long enough to pay for the larger code.
using Big = FfmaConfig<128, 128, 32, 3, 2, 2, 2, 8, 16, 4>;
using BigShortK = FfmaConfig<128, 128, 32, 3, 2, 2, 2, 8, 16, 1>;
// 256 x 128 CTA tile, 8 warps (4 x 2 of 64 x 64), 8 x 16 per thread, BK = 32, 3 stages: 144 KB
// of ring, one CTA (8 warps) per SM. The same warps per SM as two 128 x 128 CTAs, with three
// quarters of the staged bytes and half the barrier rounds per FLOP: in whole rounds 4-5 %
// faster (3072^3: 63.4 against 60.5 TFLOP/s), while its coarser rounds leave longer tails.
using Huge = FfmaConfig<256, 128, 32, 3, 4, 2, 2, 8, 16, 4>;
// The same tile with 64-deep K blocks (two 32-deep sub-blocks of A per stage) in 2 stages of
// 96 KB: half the K-block boundaries per FLOP, each of which costs every warp a barrier wait and
// the first fragment loads of the block. It runs the whole-round launches over all of K on the
// TMA path: 4096^3 65.2 -> 66.0 TFLOP/s, 3072^3 63.4 -> 64.2, 2048^3 55.4 -> 56.2, the same
// bits. The k loop is unrolled over 4 of its 8 groups: all 8 ran 56.3 at 4096^3 (the code
// outgrows the instruction cache). K ranges that end inside K and are not whole 64-deep blocks
// (TMA zero-fills only beyond K), the general path (a 2-stage ring cannot issue a stage S - 2
// blocks ahead) and the short-K kernel keep the 32-deep tile.
using Huge64 = FfmaConfig<256, 128, 64, 2, 4, 2, 2, 8, 16, 4>;
// 4 x 8 per thread (64 x 64 CTA tiles of 4 warps, BK = 32, 3 stages): many small CTAs (four
// per SM) that even out the last wave. Measured fastest up to ~2.4 tiles of 128 x 128 per SM:
// 1024^3 37.0 TFLOP/s (BK = 16 and 4 stages: 32.4; 128 x 64 tiles of 8 x 8: 35.8), 2048^3 52.3
// (128 x 128: 51.1), 2304^3 52.1 (45.9).
using Small48 = FfmaConfig<64, 64, 32, 3, 2, 2, 2, 4, 8, 1>;
// With 64-deep K blocks over all of K (3 stages of 32 KB, two CTAs per SM instead of four):
// 768^3 30.9 -> 35.1 TFLOP/s, 640^3 20.8 -> 22.6, 1280^3 44.2 -> 45.2, the 4096^3 tail 65.9 ->
// 66.0 per call. This ring depth serves the general path, which needs three stages.
using Small48K64 = FfmaConfig<64, 64, 64, 3, 2, 2, 2, 4, 8, 1>;
// On the TMA path the same tile runs 2 stages, so three CTAs fit an SM (12 warps) instead of
// two: the 448 tail tiles at 4096^3 then all run at once (456 slots) instead of in a full and a
// partial wave. 4096^3 66.1 -> 66.5 TFLOP/s, 3584^3 63.7 -> 64.1, 2560^3 60.3 -> 60.8, 1152^3
// 36.1 -> 37.0, 1280^3 45.2 -> 46.2, 640^3 and 768^3 unchanged; the same bits.
using Small48K64T = FfmaConfig<64, 64, 64, 2, 2, 2, 2, 4, 8, 1>;
// 128 x 64 tiles of 4 warps, 8 x 8 per thread (pipelined fragments): about one tile per SM.
using Tall88 = FfmaConfig<128, 64, 32, 3, 2, 2, 2, 8, 8, 1>;
// (64-deep K blocks leave one CTA per SM here, three stages of 48 KB: 1792^3 50.0 -> 47.5, so
// this tile keeps 32-deep ones.)
// Tiles of 8 warps for problems of at most one tile per SM, where a CTA runs alone on its SM
// and its latency shows: 128 x 128 of 8 x 8 per thread (1536^3: 55.9 TFLOP/s against 52.6
// with two 128 x 64 tiles per SM) and 128 x 64 of 8 x 4 per thread (1024^3: 41.4 against
// 39.9 with 4 warps of 8 x 8).
using Big88 = FfmaConfig<128, 128, 32, 3, 2, 4, 2, 8, 8, 1>;
using Tall84 = FfmaConfig<128, 64, 32, 3, 2, 4, 2, 8, 4, 1>;
// With 64-deep K blocks over all of K: 1408^3 46.7 -> 48.0 TFLOP/s, 1536^3 55.5 -> 55.9
// (128 x 128); 1152 x 1024 x 512 39.6 -> 41.2 (128 x 64).
using Big88K64 = FfmaConfig<128, 128, 64, 3, 2, 4, 2, 8, 8, 1>;
using Tall84K64 = FfmaConfig<128, 64, 64, 3, 2, 4, 2, 8, 4, 1>;
// 56 x 128 tiles of 8 warps (1 x 8 of 56 x 16), 7 x 4 per thread, A read 4 k values at a time:
// a 1024 x 1024 C is 19 x 8 = 152 of them, one per SM, where 128 x 64 tiles leave 24 SMs idle
// and give the busiest SM 14 % more work. Per SM both run the FMA pipe about 70 % busy, so the
// gain is the balance: 1024^3 44.0-45.0 TFLOP/s against 41.4, 1024^2 x 4096 50.3 against 45.9,
// 1000 x 1003 x 997 26.5 against 24.2. (Measured alongside: B read 8 bytes at a time, A 4 k
// values at a time in the 128 x 64 tile, 4 x 8 per thread in it, 120 x 64 tiles of 12 warps,
// 4 stages: none faster.)
using Wide74 = FfmaConfig<56, 128, 32, 3, 1, 8, 4, 7, 4, 1>;
// The same tile with 64-deep K blocks for launches over all of K (and K ranges that 64-deep
// blocks can tile; see launch_ffma_range): a 7 x 4 tile's short K block does not hide the
// barrier wait and the first fragment loads at each block boundary (16-deep blocks had
// measured 13.5 % slower at 1024^3). 1024^3 44.0-45.0 -> 49.2 TFLOP/s, 1024^2 x 4096 49.7 ->
// 55.0, the same bits; the ragged 1000 x 1003 x 997 (producer warps, 4 stages of 46 KB) is
// unchanged at 38.6. Unlike the other 8-warp tiles it also pays at two or more tiles per SM,
// in 2 stages (see Wide74K64T and pick_ffma).
using Wide74K64 = FfmaConfig<56, 128, 64, 3, 1, 8, 4, 7, 4, 1>;
// The same in 2 stages (94 KB), so that two CTAs share an SM, on the TMA path where the tiles
// outnumber the SMs: 1408^3 50.2 -> 52.1 TFLOP/s, 1792^3 56.6 -> 58.4, 1792^2 x 512 49.7 ->
// 53.0, 1408^2 x 512 44.4 -> 46.5, 2048 x 1024 x 2048 55.0 -> 55.7. At one tile per SM the
// CTA runs alone and keeps the deeper ring.
using Wide74K64T = FfmaConfig<56, 128, 64, 2, 1, 8, 4, 7, 4, 1>;
// 32 x 32 tiles of 4 warps, 2 x 4 per thread: for products so small that 64 x 64 tiles leave
// most SMs idle, four times as many CTAs, each with a quarter of the work. Its FMA issue rate
// is low, so it pays only while 64 x 64 tiles come to at most about half an SM each: 256^3
// 3.1 TFLOP/s against 2.6, 384^3 8.8 against 6.7, 512^3 14.1 against 12.7, 512^2 x 2048 20.7
// against 17.0; 640^3 19.2 against 20.8 and 768^3 22.9 against 33.2 (BK = 16 in 4 stages was
// slower everywhere, 32 x 64 tiles of 2 x 8 per thread no faster).
using Tiny24 = FfmaConfig<32, 32, 32, 3, 2, 2, 2, 2, 4, 1>;
// With 64-deep K blocks over all of K: 384^3 8.8 -> 10.4 TFLOP/s, 512^2 x 2048 19.9 -> 21.6.
using Tiny24K64 = FfmaConfig<32, 32, 64, 3, 2, 2, 2, 2, 4, 1>;

bool tma_ok(const Problem& p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p.A), b = reinterpret_cast<uintptr_t>(p.B);
  return p.K % 4 == 0 && p.N % 4 == 0 && (a & 15u) == 0 && (b & 15u) == 0;
}

template <class Cfg>
cudaError_t run_any(const Problem& p, int splits = 1, int k_chunk = 0, float* out = nullptr,
                    TilePart part = TilePart()) {
  return tma_ok(p) ? run<Cfg, true>(p, splits, k_chunk, out, part)
                   : run<Cfg, false>(p, splits, k_chunk, out, part);
}

// The 256 x 128 tile with 64-deep K blocks where the launch may take them (`deep64`, see
// launch_ffma_range) on the TMA path; the 32-deep configuration otherwise.
cudaError_t run_huge(const Problem& p, bool deep64, const TilePart& part) {
  if (deep64 && tma_ok(p)) return run<Huge64, true>(p, 1, 0, nullptr, part);
  return run_any<Huge>(p, 1, 0, nullptr, part);
}

// The 56 x 128 tile over all of K: 2 stages (two CTAs per SM) on the TMA path when there are
// more tiles than SMs, else 3.
cudaError_t run_wide74_whole(const Problem& p, int sms, const TilePart& part) {
  if (tma_ok(p) && ((p.M + 55) / 56) * ((p.N + 127) / 128) > sms)
    return run<Wide74K64T, true>(p, 1, 0, nullptr, part);
  return run_any<Wide74K64>(p, 1, 0, nullptr, part);
}

// The 64 x 64 tile over all of K: 2 stages on the TMA path, 3 on the general path.
cudaError_t run_small48_whole(const Problem& p, const TilePart& part) {
  if (tma_ok(p)) return run<Small48K64T, true>(p, 1, 0, nullptr, part);
  return run<Small48K64, false>(p, 1, 0, nullptr, part);
}

}  // namespace

cudaError_t launch_ffma(const Problem& p) { return launch_ffma_concurrent(p, 1); }

namespace {

// The values are those of t2s_gemm_f32_plan.
enum class FfmaPick {
  kBig = 0,
  kBigShortK = 1,
  kTall88 = 2,
  kSmall48 = 3,
  kHuge = 4,
  kHugeTail = 5,
  kBig88 = 6,
  kTall84 = 7,
  kPersistent = 8,
  kWide74 = 9,
  kTiny24 = 10,
  kPersistentStore = 11
};

// Picks the configuration whose busiest SM has the least work: ceil(tiles / SMs) tiles of the
// configuration's area, divided by its relative efficiency per FLOP, fitted to a sweep of square
// and rectangular shapes from 768 to 8192 on GB300:
//  * 64 x 64 tiles 1.0; 128 x 64 1.05; 64 x 128 1.04 (never ahead of 128 x 64, so not built);
//    32 x 32 0.6 (fitted from 256^3 to 768^3);
//  * 128 x 128 tiles 1.15 from three tiles per SM on, 1.05 at two and 1.03 at one (with the
//    compact k loop; the fully unrolled one pays only from three);
//  * 256 x 128 tiles 1.17 (K >= 256). They also run as whole rounds followed by the rest of
//    their tiles cut into 64 x 64 ones, which the tail spreads over all SMs: floor(tiles / SMs)
//    rounds plus ceil(8 x rest / SMs) small tiles;
//  * the 8-warp tiles where they come to at most one per SM: 128 x 128 1.116, 128 x 64 1.091,
//    56 x 128 1.043;
//  * the 56 x 128 tile also at two or more per SM in a launch of 64-deep K blocks (`deep64`)
//    with K >= 128, where it runs 64-deep K blocks in 2 stages, two CTAs per SM: 1.05 (1408^3 52.2
//    against 48.4 TFLOP/s for 128 x 128 tiles of 8 warps, 1792^3 58.4 against 50.5 for 128 x 64,
//    2048^3 58.1 against 56.2 and 4096 x 1024 x 4096 59.0 against 56.8 for one round of
//    256 x 128, 896 x 5760 x 256 49.0 against 42.6 for 256 x 128 with the tail; from 2304^3 on
//    the 256 x 128 tiles stay ahead, 60.4 against 59.3; level at K = 128).
// Every measured winner of the sweep is the model's pick, up to 1-2 %, including the
// non-monotone ones (1024^3 goes to 56 x 128 tiles of 8 warps, 1280^3 to 64 x 64, 1408^3 to
// 56 x 128 again, 1536^3 to 128 x 128 of 8 warps, 1792^3 and 2048^3 to 56 x 128, 3072^3 to
// 256 x 128, 2304^3, 2560^3, 4096^3 and 6144^3 to 256 x 128 with the 64 x 64 tail).
// `copies` products of this size share the GPU; they (and K < 256) keep to the one-launch
// configurations of at most 128 x 128. `cost`, when given, receives the busiest SM's work per
// k value in the model's units (area / efficiency).
// Short K: measured against the one-launch tilings (L2 flushed): 16384^2 x 32 51.1 against
// 47.6 TFLOP/s, 16384^2 x 16 25.4 against 23.5, 8192 x 4096 x 32 43.1 against 39.8, 8192^2 x
// 64 54.2 against 53.6, 6144^2 x 96 54.2 against 53.4; from K = 128 on the plain tiles win
// (8192^2 x 128: 58.1 against 59.4).
constexpr int64_t kPStoreMaxK = 96;

FfmaPick pick_ffma(int64_t M, int64_t N, int64_t K, int sms, int copies, bool deep64,
                   double* cost = nullptr) {
  struct Cand {
    FfmaPick pick;
    int bm, bn;
    double eff;
  };
  const Cand cands[4] = {{FfmaPick::kBig, 128, 128, 1.15},  // efficiency set per tiles per SM
                         {FfmaPick::kTall88, 128, 64, 1.05},
                         {FfmaPick::kSmall48, 64, 64, 1.0},
                         {FfmaPick::kTiny24, 32, 32, 0.6}};
  const int64_t n_copies = copies > 1 ? copies : 1;
  FfmaPick best = FfmaPick::kSmall48;
  double best_cost = 0.0;
  int64_t big_per_sm = 0;
  for (int i = 0; i < 4; ++i) {
    const int64_t tiles = ((M + cands[i].bm - 1) / cands[i].bm) * ((N + cands[i].bn - 1) / cands[i].bn) *
                          n_copies;
    const int64_t per_sm = (tiles + sms - 1) / sms;
    double eff = cands[i].eff;
    if (cands[i].pick == FfmaPick::kBig) {
      big_per_sm = per_sm;
      eff = per_sm >= 3 ? 1.15 : per_sm == 2 ? 1.05 : 1.03;
    }
    const double cost = static_cast<double>(per_sm) * cands[i].bm * cands[i].bn / eff;
    if (i == 0 || cost < best_cost) {
      best = cands[i].pick;
      best_cost = cost;
    }
  }
  {
    const Cand one[3] = {{FfmaPick::kBig88, 128, 128, 1.116},
                         {FfmaPick::kTall84, 128, 64, 1.091},
                         {FfmaPick::kWide74, 56, 128, 1.043}};
    for (int i = 0; i < 3; ++i) {
      const int64_t tiles = ((M + one[i].bm - 1) / one[i].bm) * ((N + one[i].bn - 1) / one[i].bn) *
                            n_copies;
      const int64_t per_sm = (tiles + sms - 1) / sms;
      const bool deep_wide =
          deep64 && n_copies == 1 && K >= 128 && one[i].pick == FfmaPick::kWide74;
      if (per_sm > 1 && !deep_wide) continue;
      const double cost = static_cast<double>(per_sm) * one[i].bm * one[i].bn /
                          (per_sm > 1 ? 1.05 : one[i].eff);
      if (cost < best_cost) {
        best = one[i].pick;
        best_cost = cost;
      }
    }
  }
  if (n_copies == 1 && K >= 256) {
    constexpr double kHugeEff = 1.17;
    const int64_t tiles = ((M + 255) / 256) * ((N + 127) / 128);
    const double per_tile = 256.0 * 128.0 / kHugeEff;
    const double whole = static_cast<double>((tiles + sms - 1) / sms) * per_tile;
    if (whole < best_cost) {
      best = FfmaPick::kHuge;
      best_cost = whole;
    }
    const int64_t rounds = tiles / sms, rest = tiles % sms;
    if (rounds >= 1 && rest > 0) {
      const double split = static_cast<double>(rounds) * per_tile +
                           static_cast<double>((8 * rest + sms - 1) / sms) * 64.0 * 64.0;
      if (split < best_cost) {
        best = FfmaPick::kHugeTail;
        best_cost = split;
      }
    }
  }
  // The 128 x 128 tile fully unrolls its k loop once K is long enough and every SM runs at
  // least three tiles.
  if (best == FfmaPick::kBig && (K < 256 || big_per_sm < 3)) best = FfmaPick::kBigShortK;
  // With a single K block per tile nothing in a CTA overlaps the load of its operands; a
  // persistent grid loads the next tile's while this one computes and stores (16384^2 x 32:
  // 47.6 against 42.3 TFLOP/s). From two K blocks on it measured slower (8192^2 x 64: 50.3
  // against 53.6).
  if (best == FfmaPick::kBigShortK && n_copies == 1 && K <= 32 && big_per_sm > 2)
    best = FfmaPick::kPersistent;
  // Short K (at most three K blocks) with at least two rounds of 256 x 128 tiles: storing C
  // takes about as long as the multiply-adds, and the persistent kernel with a TMA-store
  // epilogue overlaps the two.
  if (n_copies == 1 && K <= kPStoreMaxK &&
      ((M + 255) / 256) * ((N + 127) / 128) >= 2 * static_cast<int64_t>(sms))
    best = FfmaPick::kPersistentStore;
  if (cost != nullptr) *cost = best_cost;
  return best;
}

template <class... Ts>
cudaError_t run_pick(FfmaPick pick, const Problem& p, Ts... args) {
  switch (pick) {
    case FfmaPick::kBig: return run_any<Big>(p, args...);
    case FfmaPick::kBigShortK: return run_any<BigShortK>(p, args...);
    case FfmaPick::kTall88: return run_any<Tall88>(p, args...);
    case FfmaPick::kBig88: return run_any<Big88>(p, args...);
    case FfmaPick::kTall84: return run_any<Tall84>(p, args...);
    case FfmaPick::kWide74: return run_any<Wide74>(p, args...);
    case FfmaPick::kTiny24: return run_any<Tiny24>(p, args...);
    // The persistent grids run through their own launchers; a launch of tiles gets their tile.
    case FfmaPick::kPersistent:
    case FfmaPick::kPersistentStore: return run_any<BigShortK>(p, args...);
    default: return run_any<Small48>(p, args...);
  }
}

// 256 x 128 tiles in whole rounds over the SMs, then the rest of them as 64 x 64 tiles in a
// second launch (disjoint parts of C, so the order of the two launches changes no bit).
cudaError_t run_huge_tail(const Problem& p, int sms, const TilePart& range, bool deep64) {
  const int64_t tiles = ((p.M + 255) / 256) * ((p.N + 127) / 128);
  const int64_t main = tiles / sms * sms;
  TilePart head = range, tail = range;
  head.wbm = tail.wbm = Huge::BM;
  head.wbn = tail.wbn = Huge::BN;
  head.count = main;
  tail.off = main;
  cudaError_t e = run_huge(p, deep64, head);
  if (e != cudaSuccess) return e;
  return deep64 ? run_small48_whole(p, tail) : run_any<Small48>(p, 1, 0, nullptr, tail);
}

}  // namespace

int ffma_plan(int64_t M, int64_t N, int64_t K, int sms) {
  return static_cast<int>(pick_ffma(M, N, K, sms, 1, true));
}

cudaError_t launch_ffma_range(const Problem& p, int concurrent, int64_t k0, int64_t kc,
                              bool accumulate) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  TilePart range;
  range.k0 = k0;
  range.kc = kc;
  range.accumulate = accumulate ? 1 : 0;
  // The configuration is chosen by the K values this launch covers.
  const int64_t span = kc > 0 ? (p.K - k0 < kc ? p.K - k0 : kc) : p.K;
  // Blocks of a larger product that overlap on two streams (the host pipeline) run 128 x 128
  // tiles: their copies stagger them, so they share the GPU only in part, and the end-to-end
  // leg at 4096^3 measured 50.8 TFLOP/s with these tiles against 49.2 with the single-product
  // choice for two copies (128 x 64).
  if (concurrent > 1)
    return run_pick(span >= 256 ? FfmaPick::kBig : FfmaPick::kBigShortK, p, 1, 0, nullptr, range);
  // 64-deep K blocks where no block reads past this launch's K values: over all of K, a range
  // that ends at K (zero fill beyond K), or a range of whole 64-deep blocks (the host
  // pipeline's K chunks of 256 and 1024 values: end to end 4096^3 57.7 -> 58.0 TFLOP/s,
  // 2048^3 37.1 -> 38.5, the same bits). Other ranges keep 32-deep blocks: the last one would
  // read past the range, which the TMA unit does not zero-fill.
  const bool deep64 = kc == 0 || k0 + kc >= p.K || kc % 64 == 0;
  FfmaPick pick = pick_ffma(p.M, p.N, span, sms, 1, deep64);
  if (pick == FfmaPick::kPersistentStore) {
    // Whole products on the TMA path with an aligned C; otherwise the product's own tiles.
    if (kc == 0 && pstore_ok(p)) return launch_ffma_pstore(p);
    pick = span >= 256 ? FfmaPick::kBig : FfmaPick::kBigShortK;
  }
  if (pick == FfmaPick::kPersistent) {
    // The persistent loop covers whole products on the TMA path only.
    if (kc == 0 && tma_ok(p)) return launch_ffma_persistent(p);
    return run_pick(FfmaPick::kBigShortK, p, 1, 0, nullptr, range);
  }
  if (pick == FfmaPick::kHuge) return run_huge(p, deep64, range);
  if (pick == FfmaPick::kHugeTail) return run_huge_tail(p, sms, range, deep64);
  if (deep64) {
    switch (pick) {
      case FfmaPick::kWide74: return run_wide74_whole(p, sms, range);
      case FfmaPick::kBig88: return run_any<Big88K64>(p, 1, 0, nullptr, range);
      case FfmaPick::kTall84: return run_any<Tall84K64>(p, 1, 0, nullptr, range);
      case FfmaPick::kTiny24: return run_any<Tiny24K64>(p, 1, 0, nullptr, range);
      case FfmaPick::kSmall48: return run_small48_whole(p, range);
      default: break;
    }
  }
  return run_pick(pick, p, 1, 0, nullptr, range);
}

cudaError_t launch_ffma_concurrent(const Problem& p, int concurrent) {
  return launch_ffma_range(p, concurrent, 0, 0, false);
}

// ---------------------------------------------------------------------------- split K
namespace {

// C[i] = P_0[i] + P_1[i] + ... + P_{planes-1}[i], added in that order (deterministic).
template <int W>
__global__ void __launch_bounds__(256) reduce_planes_kernel(const float* __restrict__ P,
                                                            float* __restrict__ C, int64_t n,
                                                            int planes) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n / W;
       i += stride) {
    if constexpr (W == 4) {
      float4 acc = reinterpret_cast<const float4*>(P)[i];
      for (int z = 1; z < planes; ++z) {
        const float4 v = reinterpret_cast<const float4*>(P + static_cast<int64_t>(z) * n)[i];
        acc = make_float4(__fadd_rn(acc.x, v.x), __fadd_rn(acc.y, v.y), __fadd_rn(acc.z, v.z),
                          __fadd_rn(acc.w, v.w));
      }
      reinterpret_cast<float4*>(C)[i] = acc;
    } else {
      float acc = P[i];
      for (int z = 1; z < planes; ++z) acc = __fadd_rn(acc, P[static_cast<int64_t>(z) * n + i]);
      C[i] = acc;
    }
  }
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace

// K values per chunk: ceil(K / splits) rounded up to 32 (a whole number of K blocks of every
// configuration, so no TMA box straddles two chunks).
int64_t splitk_chunk(int64_t K, int splits) {
  const int64_t per = (K + splits - 1) / splits;
  return (per + 31) / 32 * 32;
}

// The number of chunks the automatic choice uses: the one whose modelled time is least, from
// 1 (the product alone) to 16, with chunks of at least 128 values (shorter ones spend their
// time filling the pipeline). The model is the product's own (pick_ffma): the busiest SM's
// work per k value for all chunks' tiles together, times the chunk length, plus the plane sum,
// which reads every plane and writes C once, plus the plane sum's launch (300 K work units,
// about 1.5 us: 256^3 in two chunks measured 2.6 TFLOP/s against 3.4 for the product alone
// with 32 x 32 tiles). The plane weight, 40.9 work units per kilobyte, is the
// least-squares fit of time = a x work + b x plane bytes + c to 132 measured points on GB300
// (12 shapes from 512^3 to 256^2 x 8192, 1 to 16 chunks each, L2 flushed). On those shapes the
// choice is within 3 % of the fastest count measured (1024^2 x 4096: 7 chunks, 55.5 TFLOP/s
// against 50.2 unsplit), except 256^2 x 8192 (9 chunks, 28.6 against 30.3 with 16); the
// earlier rule of about three rounds of chunk tiles on two CTA slots per SM lost 4-8 % at
// 768^3, 1024^3, 1280^3, 1536^3 and 1792^3.
int splitk_choice(int64_t M, int64_t N, int64_t K, int sms) {
  if (sms <= 0 || M <= 0 || N <= 0 || K <= 0) return 1;
  constexpr double kWorkPerKB = 40.9;
  constexpr double kPlaneSumLaunch = 3.0e5;
  double per_k = 0.0;
  pick_ffma(M, N, K, sms, 1, true, &per_k);
  double best = per_k * static_cast<double>(K);
  int best_s = 1;
  const int64_t max_s = K / 128 < 16 ? K / 128 : 16;
  for (int s = 2; s <= max_s; ++s) {
    const int64_t kc = splitk_chunk(K, s);
    const int planes = splitk_planes(K, s);
    if (planes < 2) continue;
    pick_ffma(M, N, kc, sms, planes, false, &per_k);
    const double plane_kb = static_cast<double>(planes + 1) * static_cast<double>(M) *
                            static_cast<double>(N) * 4.0 / 1000.0;
    const double t = per_k * static_cast<double>(kc) + kWorkPerKB * plane_kb + kPlaneSumLaunch;
    if (t < best) {
      best = t;
      best_s = s;
    }
  }
  return best_s;
}

int splitk_auto(int64_t M, int64_t N, int64_t K) { return splitk_choice(M, N, K, sm_count()); }

int splitk_planes(int64_t K, int splits) {
  const int64_t kc = splitk_chunk(K, splits);
  return static_cast<int>((K + kc - 1) / kc);
}

cudaError_t launch_ffma_splitk(const Problem& p, int splits, float* workspace) {
  const int64_t kc = splitk_chunk(p.K, splits);
  const int planes = splitk_planes(p.K, splits);
  if (planes <= 1) return launch_ffma(p);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // Configuration by the tiles of all chunks together, as for the unsplit product.
  const int chunk = static_cast<int>(kc);
  cudaError_t e = run_pick(pick_ffma(p.M, p.N, kc, sms, planes, false), p, planes, chunk, workspace);
  if (e != cudaSuccess) return e;
  const int64_t n = p.M * p.N;
  const bool v4 = n % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0;
  const int64_t work = v4 ? n / 4 : n;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  const int64_t blocks = (work + 255) / 256 < cap ? (work + 255) / 256 : cap;
  if (v4) reduce_planes_kernel<4><<<static_cast<unsigned>(blocks), 256, 0, p.stream>>>(workspace, p.C, n, planes);
  else reduce_planes_kernel<1><<<static_cast<unsigned>(blocks), 256, 0, p.stream>>>(workspace, p.C, n, planes);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------- stream K
namespace {

// First iteration of CTA c when `total` iterations are shared out evenly over `ctas` CTAs.
__host__ __device__ __forceinline__ int64_t sk_begin(int64_t c, int64_t total, int64_t ctas) {
  return c * total / ctas;
}

// The CTA whose share holds iteration g: the largest c with sk_begin(c) <= g.
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t g, int64_t total, int64_t ctas) {
  return ((g + 1) * ctas - 1) / total;
}

// Persistent stream-K product (TMA path), the data-parallel + stream-K hybrid of Osama et al.,
// "Stream-K: Work-centric Parallel Decomposition for Dense Matrix-Matrix Multiplication on the
// GPU" (PPoPP 2023), which is not on the source pages:
//  * tiles 0 .. dp_tiles - 1 (whole waves of G = gridDim.x tiles) run data-parallel: CTA c
//    takes tiles c, c + G, ..., so the tiles in flight at any time are neighbours in the
//    grouped order and share their A rows and B columns in L2;
//  * the iterations of the remaining tiles (tile x k block, tiles in the grouped order, k
//    blocks ascending) are shared out in equal contiguous ranges, CTA c taking the range
//    [sk_begin(c), sk_begin(c + 1)) of them after its data-parallel tiles.
// The TMA ring runs on across tiles. A tile whose k blocks all fall to one CTA is stored into
// C; otherwise the CTA's partial sums of it go to slot 0 (its first stream-K tile) or slot 1
// (its last) of its pair of BM x BN workspace tiles, and stream_fixup_kernel adds the partial
// tiles of every shared tile in k order.
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS)
    sgemm_ffma_stream_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, float* __restrict__ C,
                             float* __restrict__ partials, int M, int N, int tiles_m,
                             int tiles_n, int nkb, int dp_tiles, int64_t sk_total,
                             unsigned* status, int vec_store) {
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA = base;
  const uint32_t sB = sA + S * Cfg::A_STAGE_BYTES;
  const uint32_t sBar = sB + S * Cfg::B_STAGE_BYTES;  // full[S] (the empty[S] words are unused)
  const uint32_t sCnt = sBar + 16u * S;                // refill counters
  __shared__ int issue_tile, issue_kb;                 // next iteration to load
  auto full = [&](int s) { return sBar + 8u * s; };
  auto a_stage = [&](int s) { return sA + static_cast<uint32_t>(s) * Cfg::A_STAGE_BYTES; };
  auto b_stage = [&](int s) { return sB + static_cast<uint32_t>(s) * Cfg::B_STAGE_BYTES; };

  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  // Data-parallel tiles of this CTA, then its stream-K range.
  const int n_dp = c < dp_tiles ? (dp_tiles - c + G - 1) / G : 0;
  const int64_t sk0 = sk_begin(c, sk_total, G), sk1 = sk_begin(c + 1, sk_total, G);
  const int sk_first_tile = dp_tiles + static_cast<int>(sk0 / nkb);
  const int sk_first_kb = static_cast<int>(sk0 % nkb);
  const int count = n_dp * nkb + static_cast<int>(sk1 - sk0);  // the host keeps it < 2^31

  // Origin of tile t in the grouped order (8 tile-rows sweep the columns together).
  auto origin = [&](int tile, int& m0, int& n0) {
    constexpr int kGroup = 8;
    const int per_group = kGroup * tiles_n;
    const int first_m = (tile / per_group) * kGroup;
    const int gsz = min(tiles_m - first_m, kGroup);
    m0 = (first_m + (tile % per_group) % gsz) * Cfg::BM;
    n0 = ((tile % per_group) / gsz) * Cfg::BN;
  };
  // Loads the next iteration into ring slot s and advances the cursor. Loads are issued in
  // iteration order (the prologue, then the refill of each slot once every warp is done
  // with it, which happens in slot order), so one cursor serves all issuing threads.
  auto issue_next = [&](int s) {
    const int tile = issue_tile, kb = issue_kb;
    int m0, n0;
    origin(tile, m0, n0);
    tma_stage<Cfg>(&tmA, &tmB, m0, n0, kb * Cfg::BK, a_stage(s), b_stage(s), full(s));
    if (kb + 1 < nkb) {
      issue_kb = kb + 1;
    } else if (tile < dp_tiles && tile + G < dp_tiles) {
      issue_tile = tile + G;  // next data-parallel tile
      issue_kb = 0;
    } else if (tile < dp_tiles) {
      issue_tile = sk_first_tile;  // data-parallel part done: the stream-K range
      issue_kb = sk_first_kb;
    } else {
      issue_tile = tile + 1;
      issue_kb = 0;
    }
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1u);
      asm volatile("st.shared.u32 [%0], 0;" ::"r"(sCnt + 4u * s) : "memory");
    }
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    issue_tile = n_dp > 0 ? c : sk_first_tile;
    issue_kb = n_dp > 0 ? 0 : sk_first_kb;
    for (int j = 0; j < S && j < count; ++j) issue_next(j);
  }
  __syncthreads();

  const int wm0 = (warp % Cfg::WARPS_M) * Cfg::WM;
  const int wn0 = (warp / Cfg::WARPS_M) * Cfg::WN;
  const int g = lane >> 2, h = lane & 3;
  const uint32_t a_row0 = static_cast<uint32_t>((wm0 + g) * Cfg::A_ROW_BYTES);
  const uint32_t xr = (a_row0 >> 7) & Cfg::SWZ_MASK;
  const uint32_t b_col0 = static_cast<uint32_t>((wn0 + 4 * h) * 4);

  uint64_t acc[Cfg::TM][Cfg::TN / 2];
  int j = 0;  // local iteration
  int tile = n_dp > 0 ? c : sk_first_tile;
  int kb0 = n_dp > 0 ? 0 : sk_first_kb;
  while (j < count) {
    // This CTA's part of `tile`: k blocks kb0 .. kb0 + len - 1.
    const int len = min(nkb - kb0, count - j);
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
      for (int q = 0; q < Cfg::TN / 2; ++q) acc[i][q] = 0ull;
    for (int jend = j + len; j < jend; ++j) {
      const int s = j % S;
      const bool landed = mbar_wait_bounded(full(s), static_cast<uint32_t>(j / S) & 1u, status);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) {
          for (int q = j; q < j + S && q < count; ++q)
            mbar_wait_bounded(full(q % S), static_cast<uint32_t>(q / S) & 1u, status, 10000000ull);
        }
        return;
      }
      ffma_kblock<Cfg>(acc, a_stage(s) + a_row0, b_stage(s) + b_col0, xr);
      __syncwarp();
      if (lane == 0) {
        // The last warp to finish with this slot refills it with iteration j + S.
        if (slot_done_count(sCnt + 4u * s) == Cfg::WARPS - 1) {
          asm volatile("st.shared.u32 [%0], 0;" ::"r"(sCnt + 4u * s) : "memory");
          if (j + S < count) issue_next(s);
        }
      }
    }
    if (kb0 == 0 && len == nkb) {
      int m0, n0;
      origin(tile, m0, n0);
      store_tile<Cfg>(acc, C, M, N, m0 + wm0 + g, n0 + wn0 + 4 * h, vec_store);
    } else {
      float* slot = partials + (2 * static_cast<int64_t>(c) + (tile == sk_first_tile ? 0 : 1)) *
                                   (Cfg::BM * Cfg::BN);
      store_tile<Cfg>(acc, slot, Cfg::BM, Cfg::BN, wm0 + g, wn0 + 4 * h, 1);
    }
    if (tile < dp_tiles) {
      tile += G;
      kb0 = 0;
      if (tile >= dp_tiles) {
        tile = sk_first_tile;
        kb0 = sk_first_kb;
      }
    } else {
      ++tile;
      kb0 = 0;
    }
  }
}

// Tiles shared by several CTAs: C = P_c0 + P_c0+1 + ... + P_c1, the partial tiles of the CTAs
// that ran the tile's k blocks, added in that (ascending k) order. kFixupSplit CTAs per tile,
// each over a contiguous part of the tile in float4 groups (BN % 4 == 0); tiles run whole by
// one CTA return at once. The slots of the contributors are found once per CTA.
constexpr int kFixupSplit = 8;
constexpr int kMaxStreamCtas = 1024;

template <int BM, int BN>
__global__ void __launch_bounds__(256) stream_fixup_kernel(const float* __restrict__ partials,
                                                           float* __restrict__ C, int M, int N,
                                                           int tiles_m, int tiles_n, int nkb,
                                                           int dp_tiles, int64_t sk_total,
                                                           int64_t ctas) {
  __shared__ int slot_of[kMaxStreamCtas];
  // Stream-K tile t (tile dp_tiles + t of the grouped order).
  const int64_t t = blockIdx.x / kFixupSplit;
  const int part = static_cast<int>(blockIdx.x % kFixupSplit);
  const int64_t c0 = sk_owner(t * nkb, sk_total, ctas);
  const int64_t c1 = sk_owner((t + 1) * nkb - 1, sk_total, ctas);
  if (c0 == c1) return;
  const int n = static_cast<int>(c1 - c0 + 1);
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    const int64_t c = c0 + q;
    slot_of[q] = static_cast<int>(2 * c + (t == sk_begin(c, sk_total, ctas) / nkb ? 0 : 1));
  }
  __syncthreads();
  constexpr int kGroup = 8;
  const int tile = dp_tiles + static_cast<int>(t);
  const int per_group = kGroup * tiles_n;
  const int first_m = (tile / per_group) * kGroup;
  const int gsz = min(tiles_m - first_m, kGroup);
  const int m0 = (first_m + (tile % per_group) % gsz) * BM;
  const int n0 = ((tile % per_group) / gsz) * BN;
  constexpr int kVecs = BM * BN / 4;
  constexpr int kPer = kVecs / kFixupSplit;
  const float4* P = reinterpret_cast<const float4*>(partials);
  for (int v = part * kPer + threadIdx.x; v < (part + 1) * kPer; v += blockDim.x) {
    float4 sum = P[static_cast<int64_t>(slot_of[0]) * kVecs + v];
    for (int q = 1; q < n; ++q) {
      const float4 x = P[static_cast<int64_t>(slot_of[q]) * kVecs + v];
      sum = make_float4(__fadd_rn(sum.x, x.x), __fadd_rn(sum.y, x.y), __fadd_rn(sum.z, x.z),
                        __fadd_rn(sum.w, x.w));
    }
    const int r = (4 * v) / BN, c = (4 * v) % BN;
    const int row = m0 + r, col = n0 + c;
    if (row >= M) continue;
    float* dst = C + static_cast<int64_t>(row) * N + col;
    if (col + 0 < N) dst[0] = sum.x;
    if (col + 1 < N) dst[1] = sum.y;
    if (col + 2 < N) dst[2] = sum.z;
    if (col + 3 < N) dst[3] = sum.w;
  }
}

}  // namespace

// Partial-tile workspace of the stream-K product: two 128 x 128 tiles per CTA.
size_t streamk_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)M;
  (void)N;
  (void)K;
  const int sms = sm_count();
  return static_cast<size_t>(2 * (sms > 0 ? sms : 1)) * 2 * 128 * 128 * sizeof(float);
}

bool streamk_supported(const Problem& p) { return tma_ok(p); }

// The persistent loop of the stream-K kernel with every tile data-parallel: 2 CTAs per SM walk
// tiles c, c + G, ... of the grouped order with one TMA ring across tiles, so the next tile's
// operands load while this tile computes and stores. Each tile is summed by one CTA in
// ascending k: the bits of the product.
cudaError_t launch_ffma_persistent(const Problem& p) {
  using Cfg = BigShortK;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap ta, tb;
  cudaError_t e = encode_tmap_f32_2d(&ta, p.A, p.K, p.M, Cfg::BKS, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = encode_tmap_f32_2d(&tb, p.B, p.N, p.K, Cfg::BN, Cfg::BK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  auto kern = sgemm_ffma_stream_kernel<Cfg>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  const int64_t tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
  const int64_t tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t nkb = (p.K + Cfg::BK - 1) / Cfg::BK;
  const int64_t slots = 2 * static_cast<int64_t>(sms);
  const int64_t ctas = tiles < slots ? tiles : slots;
  if (tiles > 0x7fffffffLL || (tiles / ctas + 1) * nkb > 0x7fffffffLL)
    return cudaErrorInvalidConfiguration;
  const int vec_store = (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) ? 1 : 0;
  kern<<<static_cast<unsigned>(ctas), Cfg::THREADS, Cfg::SMEM_BYTES, p.stream>>>(
      ta, tb, p.C, nullptr, static_cast<int>(p.M), static_cast<int>(p.N),
      static_cast<int>(tiles_m), static_cast<int>(tiles_n), static_cast<int>(nkb),
      static_cast<int>(tiles), 0, p.status, vec_store);
  return cudaGetLastError();
}

// The persistent product with the TMA-store epilogue (sgemm_ffma_pstore_kernel): 256 x 128
// tiles, one CTA per SM, 2 ring stages. TMA path only, and C 16-byte aligned.
template <class Cfg, int S, int PASSES>
cudaError_t launch_pstore(const Problem& p) {
  using P = PStore<Cfg, S, PASSES>;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap ta, tb, tc;
  cudaError_t e = encode_tmap_f32_2d(&ta, p.A, p.K, p.M, Cfg::BKS, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess) e = encode_tmap_f32_2d(&tb, p.B, p.N, p.K, Cfg::BN, Cfg::BK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess) e = encode_tmap_f32_2d(&tc, p.C, p.N, p.M, 32, P::ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  auto kern = sgemm_ffma_pstore_kernel<Cfg, S, PASSES>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  const int64_t tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
  const int64_t tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
  const int64_t tiles = tiles_m * tiles_n;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int64_t slots = static_cast<int64_t>(sms) * Cfg::MIN_BLOCKS;
  const int64_t ctas = tiles < slots ? tiles : slots;
  kern<<<static_cast<unsigned>(ctas), Cfg::THREADS, P::SMEM_BYTES, p.stream>>>(
      ta, tb, tc, static_cast<int>(p.M), static_cast<int>(p.N), static_cast<int>(p.K),
      static_cast<int>(tiles_m), static_cast<int>(tiles_n), p.status);
  return cudaGetLastError();
}

// One CTA of 256 x 128 tiles per SM, staging whole warp parts. Measured alongside and not kept:
// two CTAs of 128 x 128 tiles per SM staging half a warp part at a time (so that one CTA's
// stores overlap the other's multiply-adds), 16384^2 x 32 47.5 against 51.1 TFLOP/s, 8192^2 x 64
// 49.8 against 54.2; raster groups of 1, 2 or 32 tile rows instead of 8: within 2 %; 128 x 256
// tiles (1 KB of each C row per tile instead of 512 bytes): within 1 %; warps 4-7 started 1000 to
// 4000 cycles late, so that the two warps of a sub-partition stage at different times: +1-3 %
// (the offset drifts away within a few tiles); the stores issued during the first K groups of the
// next tile: no gain at K = 32, slower from K = 64 on; a warpgroup of 4 store warps issuing them
// (setmaxnreg: 40 registers each, 232 for the compute warps): +1 % at K = 32, slower at 8192 x
// 4096 x 32 and 6144^2 x 96, the compute warps' multiply-adds 4 % slower. Per-warp cycle counts
// at 16384^2 x 32: a tile takes about 11.6 K cycles, 9.2 K of them multiply-adds and 1.45 K
// staging C and issuing its stores (all warps at once; lane 0 waits about 0.7 K while the TMA unit
// takes the boxes). C leaves the SMs at 6-7.7 TB/s at most, whatever the store pattern
// (t2s_probe_store_f32: 6.37 TB/s at 16384^2), so the 1.07 GB of C needs about 170 us against
// about 254 us of multiply-adds; K = 16 costs as much as K = 32 because the 32-deep K block is
// zero-padded.
cudaError_t launch_ffma_pstore(const Problem& p) { return launch_pstore<Huge, 2, 1>(p); }

bool pstore_ok(const Problem& p) {
  return tma_ok(p) && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0;
}

cudaError_t launch_ffma_streamk(const Problem& p, float* workspace) {
  // The compact k loop: a fully unrolled one measured slower in this persistent loop.
  using Cfg = BigShortK;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  CUtensorMap ta, tb;
  cudaError_t e = encode_tmap_f32_2d(&ta, p.A, p.K, p.M, Cfg::BKS, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = encode_tmap_f32_2d(&tb, p.B, p.N, p.K, Cfg::BN, Cfg::BK, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  auto kern = sgemm_ffma_stream_kernel<Cfg>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  const int64_t tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
  const int64_t tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t nkb = (p.K + Cfg::BK - 1) / Cfg::BK;
  if (tiles * kFixupSplit > 0x7fffffffLL || nkb > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // Two CTAs per SM (the product kernel's occupancy), each with at least 4 k blocks so that
  // small products do not split into many partial tiles.
  const int64_t slots = 2 * static_cast<int64_t>(sms);
  const int64_t by_work = (tiles * nkb + 3) / 4;
  int64_t ctas = by_work < slots ? by_work : slots;
  if (ctas > kMaxStreamCtas) ctas = kMaxStreamCtas;
  // All whole waves but the last run data-parallel; the rest (one to two waves of tiles) is
  // shared out. A tile count that is a whole number of waves runs all data-parallel.
  const int64_t waves = tiles / ctas;
  const int64_t dp_tiles = tiles % ctas == 0 ? tiles : (waves > 0 ? (waves - 1) * ctas : 0);
  const int64_t sk_tiles = tiles - dp_tiles;
  const int64_t sk_total = sk_tiles * nkb;
  const int64_t per_cta = (dp_tiles / ctas + 1) * nkb + sk_total / ctas + 1;
  if (per_cta > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int vec_store = (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) ? 1 : 0;
  kern<<<static_cast<unsigned>(ctas), Cfg::THREADS, Cfg::SMEM_BYTES, p.stream>>>(
      ta, tb, p.C, workspace, static_cast<int>(p.M), static_cast<int>(p.N),
      static_cast<int>(tiles_m), static_cast<int>(tiles_n), static_cast<int>(nkb),
      static_cast<int>(dp_tiles), sk_total, p.status, vec_store);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (sk_tiles > 0) {
    stream_fixup_kernel<Cfg::BM, Cfg::BN><<<static_cast<unsigned>(sk_tiles * kFixupSplit), 256, 0,
                                            p.stream>>>(
        workspace, p.C, static_cast<int>(p.M), static_cast<int>(p.N), static_cast<int>(tiles_m),
        static_cast<int>(tiles_n), static_cast<int>(nkb), static_cast<int>(dp_tiles), sk_total,
        ctas);
  }
  return cudaGetLastError();
}

}  // namespace t2s
