// tc_gemm.cuh -- persistent tcgen05 GEMM core shared by the 3xTF32, BF16 and FP16 products.
//
// C (FP32, row-major) = A x B with A given as M x K K-major planes and B as N x K K-major
// planes (B transposed) or, for 16-bit operands, as B itself (MN-major), staged by TMA in
// 64- or 128-byte swizzled rows, multiplied by tcgen05.mma with TMEM accumulators, and
// drained by epilogue warps that add each K chunk's partial sums into FP32 registers with
// round-to-nearest (WIDE tiles: one accumulator over all of K) and store C in swizzled
// shared-memory boxes with TMA.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "t2s_device.cuh"
#include "t2s_internal.h"
#include "t2s_tmap.h"

namespace t2s {
namespace tc {

// ------------------------------------------------------------------ tcgen05 helpers
// G = 1: the CTA's own tensor core; G = 2: a pair of CTAs (a cluster of two on two SMs) that
// allocate TMEM together and run MMAs of twice the rows, issued by the CTA of rank 0. Every
// tcgen05 instruction of a kernel uses the same G.
template <int G>
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  if constexpr (G == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int G>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (G == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  } else {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  }
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T; `accumulate` = 0 overwrites D.
// KIND 0: kind::tf32; otherwise kind::f16 (the instruction descriptor says BF16 or FP16).
template <int KIND, int G>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (KIND == 0 && G == 1) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else if constexpr (KIND == 0) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else if constexpr (G == 1) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrives once on the mbarrier when all tcgen05.mma issued so far by this thread are done.
template <int G>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  if constexpr (G == 1) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
  } else {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
  }
}

// The same, arriving on the mbarrier at offset `bar` of both CTAs of the pair.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

// Shared::cluster address of the same shared-memory offset in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrives once on an mbarrier given by its shared::cluster address (possibly another CTA's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA 2-D tile load into this CTA's shared memory whose completion is counted on an mbarrier
// of either CTA of the pair (given by its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// 16 consecutive 32-bit TMEM columns of the warp's 32 lanes: thread t gets lane base + t.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit TMEM columns of the warp's 32 lanes: thread t gets lane base + t.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ product kernel
// Operand kinds: 3xTF32 (two TF32 planes per operand, three MMAs per k step), BF16 and FP16
// (one plane per operand, one MMA per k step); all accumulate in FP32.
enum TcKind : int { kTf32x3 = 0, kBf16 = 1, kF16 = 2 };

// B_MN: B is read in its own row-major K x N layout (MN-major for the tensor core; 16-bit
// operands only) instead of as an N x K transposed plane.
// PAIR: CTAs run in clusters of two on two SMs that compute one 256-row tile together with
// tcgen05 .cta_group::2 MMAs (issued by rank 0): each CTA stages its 128 rows of A and half of
// B's columns (MN-major boxes, or BN / 2 rows of each K-major B plane), and accumulates its 128
// rows in its own TMEM. Each SM thus receives half of the B tile instead of all of it.
//
// WIDE (CTA pairs with B read in place only): the tile is twice the widest MMA, BN = 512; each
// k step issues two N = 256 MMAs into the two halves of one 512-column TMEM accumulator, so an
// SM stages 128 rows of A and 256 columns of B for 128 x 512 outputs -- a quarter fewer operand
// bytes per FLOP than 256-wide pair tiles. TMEM then holds a single accumulator: the tensor
// core sums all of K (no K chunks), and the epilogue streams it from TMEM to C.
template <int KIND_, int BN_, int BK_, int STAGES_, int CHUNK_K_, bool B_MN_ = false,
          bool PAIR_ = false, bool WIDE_ = false>
struct TcConfig {
  static constexpr int KIND = KIND_;
  static constexpr bool B_MN = B_MN_;
  static constexpr bool PAIR = PAIR_;
  static constexpr bool WIDE = WIDE_;
  static constexpr int NH = WIDE ? 2 : 1;  // MMAs per k step, along N
  static constexpr int MMA_N = BN_ / NH;
  static_assert(!WIDE || (PAIR_ && B_MN_), "wide tiles are CTA-pair tiles with B in place");
  static constexpr int BM = 128, BN = BN_, BK = BK_, STAGES = STAGES_;
  static constexpr int ELEM = KIND == kTf32x3 ? 4 : 2;    // bytes per operand element
  static constexpr int MMA_K = KIND == kTf32x3 ? 8 : 16;  // K of one instruction (32 bytes)
  static constexpr int PLANES = KIND == kTf32x3 ? 2 : 1;  // smem boxes per operand per stage
  static_assert(MMA_N % 16 == 0 && MMA_N >= 32 && MMA_N <= 256, "UMMA N for M = 128");
  // K-major A rows are staged in swizzle atoms of up to 128 bytes: a deeper K block is several
  // atom-wide TMA boxes side by side (16-bit operands with B read in place only).
  static_assert(BK * ELEM == 64 || BK * ELEM == 128 || (BK * ELEM == 256 && B_MN_),
                "64- or 128-byte swizzled K-major rows, or two 128-byte atoms");
  // K values accumulated inside the tensor core before the partial sum is added, with
  // round-to-nearest, into the FP32 sums the epilogue warps keep in registers.
  static constexpr int CHUNK_KB = WIDE ? (1 << 28) : CHUNK_K_ / BK;
  static_assert(CHUNK_K_ % BK == 0 && CHUNK_K_ / BK >= 1, "chunk of whole K blocks");
  static constexpr int ROW_BYTES = BK * ELEM;
  static constexpr int ATOM_BYTES = ROW_BYTES > 128 ? 128 : ROW_BYTES;  // swizzle row width
  static constexpr int ATOM_COLS = ATOM_BYTES / ELEM;                   // K values per atom row
  static constexpr int A_SUBS = ROW_BYTES / ATOM_BYTES;                 // A boxes per plane
  static_assert(!B_MN || (KIND != kTf32x3 && BN % 64 == 0),
                "MN-major B: 16-bit operands in whole 64-column (128-byte) swizzle atoms");
  // MN-major B arrives as BN / 64 TMA boxes of BK K-rows x 64 columns (128 bytes), one after
  // another; a box is a column of 128-byte swizzle atoms (8 K-rows x 64 columns each).
  static constexpr int B_BOX_BYTES = BK * 128;
  static constexpr int B_BOXES = B_MN ? BN / 64 : 1;
  static_assert(!PAIR || (B_MN ? B_BOXES % 2 == 0 : (BN / 2) % 8 == 0),
                "pairs split B in two: an even number of MN-major boxes, or whole 8-row groups of "
                "a K-major plane");
  static constexpr int G = PAIR ? 2 : 1;                  // CTAs per MMA
  static constexpr int B_BOXES_CTA = B_BOXES / G;          // B boxes this CTA stages
  static constexpr int A_BOX_BYTES = BM * ATOM_BYTES;
  static constexpr int A_BYTES = A_SUBS * A_BOX_BYTES;
  static constexpr int B_BYTES = BN / G * ROW_BYTES;  // this CTA's share of the B tile
  static constexpr int STAGE_BYTES = PLANES * (A_BYTES + B_BYTES);
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atom alignment");
  // Epilogue: groups of 4 warps (one per TMEM lane quarter), each group owning an equal
  // share of at most 128 of the tile's columns.
  static constexpr int EPI_GROUPS = WIDE ? 2 : (BN + 127) / 128;
  static constexpr int EPI_WARPS = 4 * EPI_GROUPS;
  static constexpr int EPI_COLS = BN / EPI_GROUPS;
  static_assert(BN % EPI_GROUPS == 0 && EPI_COLS % 16 == 0, "epilogue reads 16 columns at a time");
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  // 4 KB of staging per epilogue warp for TMA stores of C, after a 1 KB barrier area: one box
  // of 32 rows x 32 FP32 columns (128-byte swizzle) for WIDE tiles, two boxes of 32 rows x 16
  // columns (64-byte swizzle, double-buffered) otherwise.
  static constexpr int STAGING_BYTES = EPI_WARPS * 4096;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024 + STAGING_BYTES;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
  // 10 warps leave 3 warps on some SM sub-partitions: keep them within its registers.
  static constexpr int MAX_REGS = THREADS > 256 ? 168 : 255;
  // Two accumulators of BN FP32 columns each (double buffer), a power of two >= 32; WIDE: one
  // of 512.
  static constexpr uint32_t ACC_COLS =
      WIDE ? 512 : BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static constexpr int NBUF = WIDE ? 1 : 2;
  static constexpr uint32_t TMEM_COLS = NBUF * ACC_COLS;
  static constexpr int B_BOXES_HALF = B_BOXES_CTA / NH;  // this CTA's boxes per MMA half
  // Matrix-descriptor swizzle code (bits 61..63): 2 = 128-byte, 4 = 64-byte.
  static constexpr uint64_t LAYOUT = ATOM_BYTES == 128 ? 2 : 4;
  // Stride between 8-row core groups: 8 rows of one atom.
  static constexpr uint32_t SBO = 8 * ATOM_BYTES;
  // Instruction descriptor: D = F32 (bits 4..5 = 1), A and B = TF32 (2), BF16 (1) or FP16 (0)
  // at bits 7..9 and 10..12, both K-major (bits 15, 16 = 0), N >> 3 at bits 17..22, M >> 4 at
  // 24..28.
  static constexpr uint32_t FMT = KIND == kTf32x3 ? 2u : KIND == kBf16 ? 1u : 0u;
  // Bit 16 = 1: B is MN-major.
  // M of one MMA: 128 rows per CTA.
  static constexpr uint32_t IDESC = (1u << 4) | (FMT << 7) | (FMT << 10) |
                                    (static_cast<uint32_t>(B_MN ? 1u : 0u) << 16) |
                                    (static_cast<uint32_t>(MMA_N >> 3) << 17) |
                                    (static_cast<uint32_t>(G * BM >> 4) << 24);
};

// Shared-memory matrix descriptor of a K-major swizzled operand starting at `addr`:
// start address >> 4 (bits 0..13), leading-dimension offset (unused for swizzled K-major,
// 16 bytes), stride-dimension offset SBO >> 4 (bits 32..45), the fixed 0b001 at bits 46..48,
// base offset 0 (atoms are aligned to their repeat), swizzle code at bits 61..63.
template <class Cfg>
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3ffffu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(Cfg::SBO >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (Cfg::LAYOUT << 61);
}

// Descriptor of an MN-major operand in 128-byte-swizzled atoms (64 BF16 columns x 8 K-rows):
// leading-dimension offset = byte stride between atoms along N (one TMA box, BK x 128 bytes),
// stride-dimension offset = byte stride between 8-row K groups (1024). These roles were
// established on the device with a single-CTA product of known integers (the swapped
// assignment gives wrong sums).
template <class Cfg>
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3ffffu) >> 4) |
         (static_cast<uint64_t>(Cfg::B_BOX_BYTES >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Tile `t` of the grouped raster order (8 tile-rows sweep the columns together).
__device__ __forceinline__ void tile_origin(int t, int tiles_m, int tiles_n, int bm, int bn,
                                            int& m0, int& n0) {
  constexpr int kGroup = 8;
  const int per_group = kGroup * tiles_n;
  const int first_m = (t / per_group) * kGroup;
  const int gsz = min(tiles_m - first_m, kGroup);
  m0 = (first_m + (t % per_group) % gsz) * bm;
  n0 = ((t % per_group) / gsz) * bn;
}

// Persistent: CTA b takes tiles b, b + gridDim.x, ... (PAIR: cluster c takes tile pairs c,
// c + clusters, ...). Roles:
//   warp 0  TMA producer (lane 0 issues) over the ring of STAGES slots, across tiles;
//   warp 1  TMEM allocation; lane 0 issues the MMAs. Each K chunk of a tile is accumulated
//           from zero into TMEM accumulator c % 2 (c counts chunks across tiles);
//   warps 2 .. 2 + EPI_WARPS - 1  epilogue: add each chunk's partial sums into FP32
//           registers with round-to-nearest (the tensor core's own accumulation is not
//           round-to-nearest, and its error would grow with K), release the accumulator,
//           and store the sums after the tile's last chunk (WIDE: copy the one accumulator
//           out at the end of the tile), through each warp's staging boxes and TMA stores.
// Barriers: full[s] / empty[s] per ring slot; acc_full[b] (a chunk's MMAs are done) and
// acc_empty[b] (the epilogue has read it) per accumulator. A fresh barrier counts its
// "previous" phase (parity 1) as complete, so first uses wait on parity 1 and pass.
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1) __maxnreg__(Cfg::MAX_REGS)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmAb, const __grid_constant__ CUtensorMap tmAs,
                   const __grid_constant__ CUtensorMap tmBb, const __grid_constant__ CUtensorMap tmBs,
                   const __grid_constant__ CUtensorMap tmC,
                  float* __restrict__ C, int M, int N, int nkb, int tiles_m, int tiles_n,
                  unsigned* status, int vec_store, int tma_c) {
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sBar = base + S * Cfg::STAGE_BYTES;
  auto full = [&](int s) { return sBar + 8u * s; };
  auto empty = [&](int s) { return sBar + 8u * (S + s); };
  const uint32_t accFull = sBar + 16u * S;          // [2]
  const uint32_t accEmpty = accFull + 16u;          // [2]
  const uint32_t mmaDone = accEmpty + 16u;
  const uint32_t sSlot = mmaDone + 8u;              // TMEM address written by tcgen05.alloc
  const uint32_t sAbort = sSlot + 4u;
  // WIDE: the epilogue warps' TMA-store staging boxes, 1024-byte aligned after the barriers.
  const uint32_t staging = sBar + 1024u;
  auto stage = [&](int s) { return base + static_cast<uint32_t>(s) * Cfg::STAGE_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work units: single tiles, or (PAIR) 256-row tiles, rows 128 * rank .. of which belong to
  // the CTA of that rank in its cluster of two.
  const int rank = Cfg::PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit0 = Cfg::PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int unit_step = Cfg::PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int units_m = Cfg::PAIR ? (tiles_m + 1) / 2 : tiles_m;
  const int units = units_m * tiles_n;
  auto origin = [&](int u, int& m0, int& n0) {
    tile_origin(u, units_m, tiles_n, Cfg::BM, Cfg::BN, m0, n0);
    if (Cfg::PAIR) m0 = m0 * 2 + rank * Cfg::BM;
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accFull + 8u * b, 1);
      // Lane 0 of each epilogue warp (PAIR: of both CTAs; only rank 0's barrier is used).
      mbar_init(accEmpty + 8u * b, Cfg::G * Cfg::EPI_WARPS);
    }
    mbar_init(mmaDone, 1);
    asm volatile("st.shared.u32 [%0], 0;" ::"r"(sAbort) : "memory");
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmAb);
    tma_prefetch_desc(&tmBb);
    if (Cfg::PLANES == 2) {
      tma_prefetch_desc(&tmAs);
      tma_prefetch_desc(&tmBs);
    }
  }
  if (warp == 1) tmem_alloc<Cfg::G>(sSlot, Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  // The peer CTA's copies, commits and arrivals target this CTA's barriers: initialise them
  // first.
  if constexpr (Cfg::PAIR) cluster_sync_all();
  tc_fence_after();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(sSlot) : "memory");

  auto aborted = [&]() {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(sAbort) : "memory");
    return v != 0u;
  };
  auto set_abort = [&]() { asm volatile("st.volatile.shared.u32 [%0], 1;" ::"r"(sAbort) : "memory"); };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (lane 0 issues)
    if (lane == 0) {
      int64_t g = 0;  // running K-block index over all tiles of this CTA
      bool ok = true;
      for (int u = unit0; ok && u < units; u += unit_step) {
        int m0, n0;
        origin(u, m0, n0);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = static_cast<int>(g % S);
          const uint32_t par = (static_cast<uint32_t>(g / S) & 1u) ^ 1u;
          if (aborted() || !mbar_wait_bounded(empty(s), par, status)) {
            set_abort();
            ok = false;
            break;
          }
          const uint32_t st = stage(s);
          const int k0 = kb * Cfg::BK;
          // Stage layout: A planes, then B planes.
          if constexpr (Cfg::PAIR) {
            // Both CTAs' copies complete on rank 0's barrier, where the MMAs wait.
            const uint32_t bar0 = map_to_rank(full(s), 0);
            if (rank == 0) mbar_arrive_expect_tx(full(s), 2 * Cfg::STAGE_BYTES);
#pragma unroll
            for (int q = 0; q < Cfg::A_SUBS; ++q)
              tma_load_2d_pair(st + q * Cfg::A_BOX_BYTES, &tmAb, k0 + q * Cfg::ATOM_COLS, m0, bar0);
            if constexpr (Cfg::B_MN) {
              // This CTA's half of each MMA's columns: box j of half h holds columns
              // h MMA_N + rank MMA_N / 2 + 64 (j % B_BOXES_HALF) .. + 63.
#pragma unroll
              for (int j = 0; j < Cfg::B_BOXES_CTA; ++j)
                tma_load_2d_pair(st + Cfg::A_BYTES + j * Cfg::B_BOX_BYTES, &tmBb,
                                 n0 + (j / Cfg::B_BOXES_HALF) * Cfg::MMA_N +
                                     (Cfg::MMA_N / 2) * rank + 64 * (j % Cfg::B_BOXES_HALF),
                                 k0, bar0);
            } else {
              // K-major B planes: this CTA's BN / 2 rows (columns of B), n0 + rank BN / 2 ..
              const int nb0 = n0 + rank * (Cfg::BN / 2);
              tma_load_2d_pair(st + Cfg::PLANES * Cfg::A_BYTES, &tmBb, k0, nb0, bar0);
              if constexpr (Cfg::PLANES == 2) {
                tma_load_2d_pair(st + Cfg::A_BYTES, &tmAs, k0, m0, bar0);
                tma_load_2d_pair(st + 2 * Cfg::A_BYTES + Cfg::B_BYTES, &tmBs, k0, nb0, bar0);
              }
            }
            continue;
          }
          mbar_arrive_expect_tx(full(s), Cfg::STAGE_BYTES);
#pragma unroll
          for (int q = 0; q < Cfg::A_SUBS; ++q)
            tma_load_2d(st + q * Cfg::A_BOX_BYTES, &tmAb, k0 + q * Cfg::ATOM_COLS, m0, full(s));
          if constexpr (Cfg::B_MN) {
#pragma unroll
            for (int j = 0; j < Cfg::B_BOXES; ++j)
              tma_load_2d(st + Cfg::A_BYTES + j * Cfg::B_BOX_BYTES, &tmBb, n0 + 64 * j, k0, full(s));
          } else {
            tma_load_2d(st + Cfg::PLANES * Cfg::A_BYTES, &tmBb, k0, n0, full(s));
          }
          if (Cfg::PLANES == 2) {
            tma_load_2d(st + Cfg::A_BYTES, &tmAs, k0, m0, full(s));
            tma_load_2d(st + 2 * Cfg::A_BYTES + Cfg::B_BYTES, &tmBs, k0, n0, full(s));
          }
        }
      }
      // Do not leave while copies into this CTA's shared memory are in flight (PAIR: while
      // they may still be unread by the MMAs; rank 0's commits free both CTAs' slots).
      for (int64_t j = g > S ? g - S : 0; j < g; ++j) {
        const int s = static_cast<int>(j % S);
        const uint32_t par = static_cast<uint32_t>(j / S) & 1u;
        if (!mbar_wait_bounded(Cfg::PAIR ? empty(s) : full(s), par, status)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (lane 0 of rank 0 issues)
    if (lane == 0 && rank == 0) {
      int64_t g = 0;   // K blocks consumed (ring position)
      int64_t cc = 0;  // chunks issued (accumulator double buffer)
      bool ok = true;
      for (int u = unit0; ok && u < units; u += unit_step) {
        for (int kb0 = 0; ok && kb0 < nkb; kb0 += Cfg::CHUNK_KB, ++cc) {
          const int b = static_cast<int>(cc % Cfg::NBUF);
          const uint32_t acc = tmem + static_cast<uint32_t>(b) * Cfg::ACC_COLS;
          // The epilogue must have read this accumulator's previous chunk.
          if (aborted() ||
              !mbar_wait_bounded(accEmpty + 8u * b,
                                 (static_cast<uint32_t>(cc / Cfg::NBUF) & 1u) ^ 1u, status)) {
            set_abort();
            ok = false;
            break;
          }
          tc_fence_after();
          const int kb1 = min(kb0 + Cfg::CHUNK_KB, nkb);
          for (int kb = kb0; kb < kb1; ++kb, ++g) {
            const int s = static_cast<int>(g % S);
            if (aborted() || !mbar_wait_bounded(full(s), static_cast<uint32_t>(g / S) & 1u, status)) {
              set_abort();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = stage(s);
#pragma unroll
            for (int k = 0; k < Cfg::BK / Cfg::MMA_K; ++k) {
              const uint32_t off = k * Cfg::MMA_K * Cfg::ELEM;  // 32 bytes per k step
              // A: the atom box holding this k step, 32-byte offset inside its rows.
              const uint64_t a_big = smem_desc<Cfg>(st + (off / Cfg::ATOM_BYTES) * Cfg::A_BOX_BYTES +
                                                    off % Cfg::ATOM_BYTES);
              // MN-major B: a k step is MMA_K whole 128-byte K-rows further on.
              const uint64_t b_big =
                  Cfg::B_MN ? smem_desc_mn<Cfg>(st + Cfg::A_BYTES + k * Cfg::MMA_K * 128)
                            : smem_desc<Cfg>(st + Cfg::PLANES * Cfg::A_BYTES + off);
              // The chunk's first MMA overwrites the accumulator (starts the partial sum at 0).
              const uint32_t acc_in = (kb != kb0 || k != 0) ? 1u : 0u;
              if constexpr (Cfg::KIND == kTf32x3) {
                const uint64_t a_small = smem_desc<Cfg>(st + Cfg::A_BYTES + off);
                const uint64_t b_small = smem_desc<Cfg>(st + 2 * Cfg::A_BYTES + Cfg::B_BYTES + off);
                mma_issue<Cfg::KIND, Cfg::G>(acc, a_small, b_big, Cfg::IDESC, acc_in);
                mma_issue<Cfg::KIND, Cfg::G>(acc, a_big, b_small, Cfg::IDESC, 1u);
                mma_issue<Cfg::KIND, Cfg::G>(acc, a_big, b_big, Cfg::IDESC, 1u);
              } else if constexpr (Cfg::WIDE) {
                // Two MMAs, one per half of the tile's columns (TMEM columns h MMA_N ..).
#pragma unroll
                for (int h = 0; h < Cfg::NH; ++h)
                  mma_issue<Cfg::KIND, Cfg::G>(
                      acc + static_cast<uint32_t>(h * Cfg::MMA_N), a_big,
                      smem_desc_mn<Cfg>(st + Cfg::A_BYTES + h * Cfg::B_BOXES_HALF * Cfg::B_BOX_BYTES +
                                        k * Cfg::MMA_K * 128),
                      Cfg::IDESC, acc_in);
              } else {
                mma_issue<Cfg::KIND, Cfg::G>(acc, a_big, b_big, Cfg::IDESC, acc_in);
              }
            }
            // Frees the ring slot when these MMAs are done (PAIR: in both CTAs).
            if constexpr (Cfg::PAIR) {
              mma_commit_pair(empty(s));
            } else {
              mma_commit<1>(empty(s));
            }
          }
          // The chunk's partial sums are complete (PAIR: in both CTAs' TMEM).
          if (ok) {
            if constexpr (Cfg::PAIR) {
              mma_commit_pair(accFull + 8u * b);
            } else {
              mma_commit<1>(accFull + 8u * b);
            }
          }
        }
      }
      // Every MMA issued above must finish before TMEM can be released.
      mma_commit<Cfg::G>(mmaDone);
      mbar_wait_bounded(mmaDone, 0u, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue: TMEM -> FP32 sums -> C
    const int e = warp - 2;
    const int q = warp & 3;                        // TMEM lanes 32q .. 32q + 31 (rows)
    const int col_base = (e >> 2) * Cfg::EPI_COLS;  // this warp's columns of the tile
    int64_t cc = 0;
    uint32_t n_boxes = 0;  // boxes this warp has stored from its staging buffer
    bool ok = true;
    for (int u = unit0; ok && u < units; u += unit_step) {
      int m0, n0;
      origin(u, m0, n0);
      if constexpr (Cfg::WIDE) {
        // The single accumulator holds the tile's sums over all of K: stream it to C.
        const bool done = !aborted() &&
                          mbar_wait_bounded(accFull, static_cast<uint32_t>(cc) & 1u, status);
        ++cc;
        if (!__all_sync(0xffffffffu, done)) {
          if (lane == 0) set_abort();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                               static_cast<uint32_t>(col_base);
        if (tma_c) {
          // 32 x 32 boxes through this warp's staging buffer: row `lane` in 128-byte-swizzled
          // order (16-byte chunk k of row r at chunk k ^ (r % 8), conflict-free per 8 lanes),
          // then one TMA store per box; the TMA unit clips what lies outside C.
          const uint32_t stg = staging + static_cast<uint32_t>(e) * 4096u;
          for (int c = 0; c < Cfg::EPI_COLS; c += 32) {
            uint32_t r[32];
            tmem_ld32(tbase + static_cast<uint32_t>(c), r);  // whole warp
            const int bx = n0 + col_base + c, by = m0 + 32 * q;  // the same for the whole warp
            if (bx >= N || by >= M) continue;
            if (lane == 0) bulk_wait_read_all();  // the previous box has left the buffer
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              st_shared_v4(stg + static_cast<uint32_t>(lane) * 128u +
                               (static_cast<uint32_t>(k ^ (lane & 7)) << 4),
                           r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tma_store_2d(&tmC, stg, bx, by);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_to_rank(accEmpty, 0));
          continue;
        }
        const int row = m0 + 32 * q + lane;
        float* crow = C + static_cast<int64_t>(row < M ? row : 0) * N;
        const int col0 = n0 + col_base;
#pragma unroll 2
        for (int c = 0; c < Cfg::EPI_COLS; c += 16) {
          uint32_t r[16];
          tmem_ld16(tbase + static_cast<uint32_t>(c), r);  // whole warp
          if (row < M) {
#pragma unroll
            for (int v = 0; v < 16; v += 4) {
              const int col = col0 + c + v;
              if (vec_store && col + 4 <= N) {
                *reinterpret_cast<float4*>(crow + col) =
                    make_float4(__uint_as_float(r[v]), __uint_as_float(r[v + 1]),
                                __uint_as_float(r[v + 2]), __uint_as_float(r[v + 3]));
              } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  if (col + i < N) crow[col + i] = __uint_as_float(r[v + i]);
              }
            }
          }
        }
        // All of this warp's TMEM reads are complete (tcgen05.ld waited).
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_rank(accEmpty, 0));  // rank 0 issues the MMAs
        continue;
      } else {
      float sum[Cfg::EPI_COLS];
#pragma unroll
      for (int c = 0; c < Cfg::EPI_COLS; ++c) sum[c] = 0.0f;
      for (int kb0 = 0; kb0 < nkb; kb0 += Cfg::CHUNK_KB, ++cc) {
        const int b = static_cast<int>(cc % Cfg::NBUF);
        const bool done = !aborted() &&
                          mbar_wait_bounded(accFull + 8u * b,
                                            static_cast<uint32_t>(cc / Cfg::NBUF) & 1u, status);
        if (!__all_sync(0xffffffffu, done)) {
          if (lane == 0) set_abort();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                               static_cast<uint32_t>(b) * Cfg::ACC_COLS +
                               static_cast<uint32_t>(col_base);
#pragma unroll
        for (int c = 0; c < Cfg::EPI_COLS; c += 16) {
          uint32_t r[16];
          tmem_ld16(tbase + static_cast<uint32_t>(c), r);
#pragma unroll
          for (int i = 0; i < 16; ++i) sum[c + i] = __fadd_rn(sum[c + i], __uint_as_float(r[i]));
        }
        // All of this warp's TMEM reads of accumulator b are complete (tcgen05.ld waited).
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (Cfg::PAIR) {
            mbar_arrive_cluster(map_to_rank(accEmpty + 8u * b, 0));  // rank 0 issues the MMAs
          } else {
            mbar_arrive(accEmpty + 8u * b);
          }
        }
      }
      if (!ok) break;
      if (tma_c) {
        // 32 x 16 boxes through the two 2 KB halves of this warp's staging buffer, taken in
        // turn by the boxes it stores (64-byte swizzle: 16-byte chunk k of row r at chunk
        // k ^ ((r / 2) % 4), conflict-free per 8 lanes), one TMA store each. Boxes wholly
        // outside C are skipped; the TMA unit clips the others at its edges.
#pragma unroll
        for (int c = 0; c < Cfg::EPI_COLS; c += 16) {
          const int bx = n0 + col_base + c, by = m0 + 32 * q;  // the same for the whole warp
          if (bx >= N || by >= M) continue;
          const uint32_t stg = staging + static_cast<uint32_t>(e) * 4096u +
                               static_cast<uint32_t>(n_boxes & 1) * 2048u;
          ++n_boxes;
          // The box stored from this half two stores ago has been read out of it.
          if (lane == 0) bulk_wait_read_but_one();
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_shared_v4(stg + static_cast<uint32_t>(lane) * 64u +
                             (static_cast<uint32_t>(k ^ ((lane >> 1) & 3)) << 4),
                         __float_as_uint(sum[c + 4 * k]), __float_as_uint(sum[c + 4 * k + 1]),
                         __float_as_uint(sum[c + 4 * k + 2]), __float_as_uint(sum[c + 4 * k + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tma_store_2d(&tmC, stg, bx, by);
        }
        continue;
      }
      const int row = m0 + 32 * q + lane;
      if (row < M) {
        float* crow = C + static_cast<int64_t>(row) * N;
        const int col0 = n0 + col_base;
#pragma unroll
        for (int c = 0; c < Cfg::EPI_COLS; c += 4) {
          if (vec_store && col0 + c + 4 <= N) {
            *reinterpret_cast<float4*>(crow + col0 + c) =
                make_float4(sum[c], sum[c + 1], sum[c + 2], sum[c + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (col0 + c + i < N) crow[col0 + c + i] = sum[c + i];
          }
        }
      }
      }
    }
    // Stores in flight read this CTA's shared memory: let them finish before it is released.
    if (tma_c && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA of a pair may exit, or release TMEM, while the other can still use its shared
  // memory, its barriers or its TMEM.
  if constexpr (Cfg::PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<Cfg::G>(tmem, Cfg::TMEM_COLS);
  }
}

// Runs the product over operand planes (K-major, `lda` / `ldb` elements per row, K padded or
// not): a0/b0 the (big) planes, a1/b1 the small planes for 3xTF32 (ignored for BF16). Every
// row stride must be a multiple of 16 bytes; K beyond the plane width reads as zeros. With
// Cfg::B_MN, b0 is B itself, K rows of `ldb` (= N) elements. `Kp` is K rounded up to BK.
template <class Cfg>
cudaError_t run_tc(const Problem& p, const void* a0, const void* a1, const void* b0,
                   const void* b1, int64_t lda, int64_t ldb, int64_t Kp) {
  CUtensorMap tAb, tAs, tBb, tBs;
  memset(&tAs, 0, sizeof(tAs));
  memset(&tBs, 0, sizeof(tBs));
  const CUtensorMapSwizzle sw =
      Cfg::ATOM_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  // TMA moves 16-bit elements as they are, so one 16-bit map type serves BF16 and FP16.
  auto enc = [&](CUtensorMap* m, const void* base, int64_t cols, int64_t rows, uint32_t box_rows) {
    return Cfg::KIND == kTf32x3
               ? encode_tmap_f32_2d(m, base, cols, rows, Cfg::ATOM_COLS, box_rows, sw)
               : encode_tmap_bf16_2d(m, base, cols, rows, Cfg::ATOM_COLS, box_rows, sw);
  };
  cudaError_t e;
  if ((e = enc(&tAb, a0, lda, p.M, Cfg::BM)) != cudaSuccess) return e;
  if constexpr (Cfg::B_MN) {
    if ((e = encode_tmap_bf16_2d(&tBb, b0, ldb, p.K, 64, Cfg::BK, CU_TENSOR_MAP_SWIZZLE_128B)) !=
        cudaSuccess)
      return e;
  } else {
    // K-major B: each CTA of a pair stages half of the tile's rows of each plane.
    if ((e = enc(&tBb, b0, ldb, p.N, Cfg::BN / Cfg::G)) != cudaSuccess) return e;
  }
  if (Cfg::PLANES == 2) {
    if ((e = enc(&tAs, a1, lda, p.M, Cfg::BM)) != cudaSuccess) return e;
    if ((e = enc(&tBs, b1, ldb, p.N, Cfg::BN / Cfg::G)) != cudaSuccess) return e;
  }
  // C as a TMA store target: row stride a multiple of 16 bytes, 16-byte aligned.
  CUtensorMap tC;
  memset(&tC, 0, sizeof(tC));
  int tma_c = 0;
  if (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) {
    if ((e = encode_tmap_f32_2d(&tC, p.C, p.N, p.M, Cfg::WIDE ? 32 : 16, 32,
                                Cfg::WIDE ? CU_TENSOR_MAP_SWIZZLE_128B
                                          : CU_TENSOR_MAP_SWIZZLE_64B)) != cudaSuccess)
      return e;
    tma_c = 1;
  }
  auto kern = tc_gemm_kernel<Cfg>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::SMEM_BYTES)) != cudaSuccess)
    return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
  const int64_t tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
  const int64_t tiles = tiles_m * tiles_n;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int vec_store = (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) ? 1 : 0;
  const int M32 = static_cast<int>(p.M), N32 = static_cast<int>(p.N);
  // K blocks over the padded K (TMA fills zeros beyond the matrices' K).
  const int nkb = static_cast<int>((Kp + Cfg::BK - 1) / Cfg::BK), tm = static_cast<int>(tiles_m),
            tn = static_cast<int>(tiles_n);
  if constexpr (Cfg::PAIR) {
    // One cluster of two CTAs per 256-row tile, at most as many clusters as can be resident
    // at once (persistent).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = p.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t units = ((tiles_m + 1) / 2) * tiles_n;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (units < sms / 2 ? units : sms / 2)));
    int resident = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&resident, kern, &cfg)) != cudaSuccess) return e;
    if (resident < 1) return cudaErrorInvalidConfiguration;
    const int64_t clusters = units < resident ? units : resident;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    return cudaLaunchKernelEx(&cfg, kern, tAb, tAs, tBb, tBs, tC, p.C, M32, N32, nkb, tm, tn,
                              p.status, vec_store, tma_c);
  } else {
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, p.stream>>>(tAb, tAs, tBb, tBs, tC, p.C, M32,
                                                            N32, nkb, tm, tn, p.status, vec_store,
                                                            tma_c);
    return cudaGetLastError();
  }
}


}  // namespace tc
}  // namespace t2s
