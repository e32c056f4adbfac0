// gemm_tf32x3.cu -- C = A x B in FP32 on the tcgen05 tensor cores with 3xTF32 error
// compensation (Ootomo and Yokota, "Recovering single precision accuracy from Tensor Cores
// while surpassing the FP32 theoretical peak performance", 2022). Not on the pages; the
// operation is the same C = A x B as the product kernel.
//
// 1. Split pre-pass (two bandwidth-bound kernels). Every x of A and B becomes
//      big = tf32(x), small = tf32(x - big)      (x - big is exact in FP32)
//    with tf32() = round to nearest even at 10 explicit mantissa bits (IEEE 754
//    rounding applied to the TF32 format, written from the definition below). The planes
//    are K-major with a padded row length Kp = ceil(K / 32) * 32 and zeros in the padding:
//      A_big, A_small : M x Kp      (A is already K-major: a row-wise copy)
//      B_big, B_small : N x Kp      (B is K x N row-major: transposed through shared memory)
//    so that every tensor-map stride is a multiple of 128 bytes whatever K and N are.
// 2. Product kernel, persistent: one CTA of 192 threads per SM walks 128 x BN tiles of C.
//      warp 0     -- TMA producer: per K block, one box of each of the four planes;
//      warp 1     -- allocates TMEM, one lane issues tcgen05.mma kind::tf32 (M=128, N=BN,
//                    K=8), three per k step into one FP32 accumulator in TMEM, in the order
//                    small*big, big*small, big*big; tcgen05.commit frees each ring slot;
//      warps 2..  -- epilogue: tcgen05.ld of their 32 TMEM lanes (rows), stores to C.
//    TMEM holds two accumulators. The tensor core accumulates one K chunk (256 values) from
//    zero; the epilogue warps add each chunk's partial sums into FP32 registers with
//    round-to-nearest while the next chunk's MMAs run. The tensor core's internal FP32
//    accumulation does not round to nearest: summed over all of K in TMEM its error grows
//    faster than K and leaves the 1e-6 K max|a| max|b| bound at K = 8192; chunking keeps
//    that error to 256 values and lets it average out across chunks.
//    Shared-memory operands use the canonical K-major layout with the 128-byte (BK = 32) or
//    64-byte (BK = 16) swizzle the TMA writes, described to the tensor core by matrix
//    descriptors.
// The missing small*small term is below 2^-22 relative; the tensor core's own summation
// order within a chunk makes the result differ from the FP32 definition by rounding only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "t2s_device.cuh"
#include "t2s_internal.h"
#include "t2s_tmap.h"

namespace t2s {
namespace {

constexpr int64_t kKPad = 32;

int64_t padded_k(int64_t K) { return (K + kKPad - 1) / kKPad * kKPad; }

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// ------------------------------------------------------------------ split pre-pass
// Round a binary32 value to the TF32 format (1 sign, 8 exponent, 10 mantissa bits), round
// to nearest, ties to even, by integer arithmetic on the encoding: add half an ulp of the
// 10-bit mantissa (minus one, plus the lowest kept bit for the tie rule) and clear the 13
// dropped bits. A carry out of the mantissa correctly increments the exponent. NaN and
// infinity are passed through.
__device__ __forceinline__ float tf32_round(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7f800000u) == 0x7f800000u) return x;
  u += 0x00000fffu + ((u >> 13) & 1u);
  return __uint_as_float(u & 0xffffe000u);
}

__device__ __forceinline__ void split(float x, float& big, float& small) {
  big = tf32_round(x);
  // x - big is exact; for non-finite x the correction term is dropped.
  small = isfinite(x) ? tf32_round(__fsub_rn(x, big)) : 0.0f;
}

// A (M x K, row-major) -> big, small (M x Kp), zeros for k >= K. Four k per thread.
__global__ void __launch_bounds__(256) split_rows_kernel(const float* __restrict__ A,
                                                         float* __restrict__ big,
                                                         float* __restrict__ small, int64_t M,
                                                         int64_t K, int64_t Kp) {
  const int64_t q = Kp / 4;
  const int64_t total = M * q;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = idx / q;
    const int64_t k = (idx % q) * 4;
    float b[4], s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = (k + e < K) ? A[row * K + k + e] : 0.0f;
      split(x, b[e], s[e]);
    }
    *reinterpret_cast<float4*>(big + row * Kp + k) = make_float4(b[0], b[1], b[2], b[3]);
    *reinterpret_cast<float4*>(small + row * Kp + k) = make_float4(s[0], s[1], s[2], s[3]);
  }
}

// B (K x N, row-major) -> big, small (N x Kp): transposed in 32 x 32 tiles through shared
// memory so that both the reads (along n) and the writes (along k) are coalesced.
__global__ void __launch_bounds__(256) split_transpose_kernel(const float* __restrict__ B,
                                                              float* __restrict__ big,
                                                              float* __restrict__ small,
                                                              int64_t K, int64_t N, int64_t Kp) {
  __shared__ float tile[32][33];
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 32;
  for (int64_t kt = blockIdx.y; kt * 32 < Kp; kt += gridDim.y) {
    const int64_t k0 = kt * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t k = k0 + ty + 8 * i, n = n0 + tx;
      tile[ty + 8 * i][tx] = (k < K && n < N) ? B[k * N + n] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = n0 + ty + 8 * i, k = k0 + tx;
      if (n < N) {
        float b, s;
        split(tile[tx][ty + 8 * i], b, s);
        big[n * Kp + k] = b;
        small[n * Kp + k] = s;
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ tcgen05 helpers
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major; `accumulate` = 0 overwrites D.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier when all tcgen05.mma issued so far by this thread are done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
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
template <int BN_, int BK_, int STAGES_, int CHUNK_K_>
struct Tf32Config {
  static constexpr int BM = 128, BN = BN_, BK = BK_, STAGES = STAGES_;
  static constexpr int MMA_K = 8;  // K of one kind::tf32 instruction
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "UMMA N for M = 128");
  static_assert(BK == 16 || BK == 32, "64- or 128-byte swizzled K-major rows");
  // K values accumulated inside the tensor core before the partial sum is added, with
  // round-to-nearest, into the FP32 sums the epilogue warps keep in registers.
  static constexpr int CHUNK_KB = CHUNK_K_ / BK;
  static_assert(CHUNK_K_ % BK == 0 && CHUNK_KB >= 1, "chunk of whole K blocks");
  static constexpr int ROW_BYTES = BK * 4;
  static constexpr int A_BYTES = BM * ROW_BYTES;
  static constexpr int B_BYTES = BN * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atom alignment");
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  // Epilogue: groups of 4 warps (one per TMEM lane quarter), each group owning an equal
  // share of at most 128 of the tile's columns.
  static constexpr int EPI_GROUPS = (BN + 127) / 128;
  static constexpr int EPI_WARPS = 4 * EPI_GROUPS;
  static constexpr int EPI_COLS = BN / EPI_GROUPS;
  static_assert(BN % EPI_GROUPS == 0 && EPI_COLS % 16 == 0, "epilogue reads 16 columns at a time");
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  // 10 warps leave 3 warps on some SM sub-partitions: keep them within its registers.
  static constexpr int MAX_REGS = THREADS > 256 ? 168 : 255;
  // Two accumulators of BN FP32 columns each (double buffer), a power of two >= 32.
  static constexpr uint32_t ACC_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
  // Matrix-descriptor swizzle code (bits 61..63): 2 = 128-byte, 4 = 64-byte.
  static constexpr uint64_t LAYOUT = BK == 32 ? 2 : 4;
  // Stride between 8-row core groups: 8 rows of ROW_BYTES.
  static constexpr uint32_t SBO = 8 * ROW_BYTES;
  // Instruction descriptor: D = F32 (bits 4..5 = 1), A and B = TF32 (bits 7..9 and 10..12 =
  // 2), both K-major (bits 15, 16 = 0), N >> 3 at bits 17..22, M >> 4 at bits 24..28.
  static constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                                    (static_cast<uint32_t>(BN >> 3) << 17) |
                                    (static_cast<uint32_t>(BM >> 4) << 24);
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

// Persistent: CTA b takes tiles b, b + gridDim.x, ... Roles:
//   warp 0  TMA producer (lane 0 issues) over the ring of STAGES slots, across tiles;
//   warp 1  TMEM allocation; lane 0 issues the MMAs. Each K chunk of a tile is accumulated
//           from zero into TMEM accumulator c % 2 (c counts chunks across tiles);
//   warps 2 .. 2 + EPI_WARPS - 1  epilogue: add each chunk's partial sums into FP32
//           registers with round-to-nearest (the tensor core's own accumulation is not
//           round-to-nearest, and its error would grow with K), release the accumulator,
//           and store the sums after the tile's last chunk.
// Barriers: full[s] / empty[s] per ring slot; acc_full[b] (a chunk's MMAs are done) and
// acc_empty[b] (the epilogue has read it) per accumulator. A fresh barrier counts its
// "previous" phase (parity 1) as complete, so first uses wait on parity 1 and pass.
template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1) __maxnreg__(Cfg::MAX_REGS)
    tf32x3_kernel(const __grid_constant__ CUtensorMap tmAb, const __grid_constant__ CUtensorMap tmAs,
                  const __grid_constant__ CUtensorMap tmBb, const __grid_constant__ CUtensorMap tmBs,
                  float* __restrict__ C, int M, int N, int nkb, int tiles_m, int tiles_n,
                  unsigned* status, int vec_store) {
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
  auto stage = [&](int s) { return base + static_cast<uint32_t>(s) * Cfg::STAGE_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = tiles_m * tiles_n;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accFull + 8u * b, 1);
      mbar_init(accEmpty + 8u * b, Cfg::EPI_WARPS);  // lane 0 of each epilogue warp
    }
    mbar_init(mmaDone, 1);
    asm volatile("st.shared.u32 [%0], 0;" ::"r"(sAbort) : "memory");
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmAb);
    tma_prefetch_desc(&tmAs);
    tma_prefetch_desc(&tmBb);
    tma_prefetch_desc(&tmBs);
  }
  if (warp == 1) tmem_alloc(sSlot, Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
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
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        int m0, n0;
        tile_origin(t, tiles_m, tiles_n, Cfg::BM, Cfg::BN, m0, n0);
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
          mbar_arrive_expect_tx(full(s), Cfg::STAGE_BYTES);
          tma_load_2d(st, &tmAb, k0, m0, full(s));
          tma_load_2d(st + Cfg::A_BYTES, &tmAs, k0, m0, full(s));
          tma_load_2d(st + 2 * Cfg::A_BYTES, &tmBb, k0, n0, full(s));
          tma_load_2d(st + 2 * Cfg::A_BYTES + Cfg::B_BYTES, &tmBs, k0, n0, full(s));
        }
      }
      // Do not leave while copies into this CTA's shared memory are in flight.
      for (int64_t j = g > S ? g - S : 0; j < g; ++j)
        if (!mbar_wait_bounded(full(static_cast<int>(j % S)), static_cast<uint32_t>(j / S) & 1u,
                               status))
          break;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (lane 0 issues)
    if (lane == 0) {
      int64_t g = 0;   // K blocks consumed (ring position)
      int64_t cc = 0;  // chunks issued (accumulator double buffer)
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        for (int kb0 = 0; ok && kb0 < nkb; kb0 += Cfg::CHUNK_KB, ++cc) {
          const int b = static_cast<int>(cc & 1);
          const uint32_t acc = tmem + static_cast<uint32_t>(b) * Cfg::ACC_COLS;
          // The epilogue must have read this accumulator's previous chunk.
          if (aborted() ||
              !mbar_wait_bounded(accEmpty + 8u * b, (static_cast<uint32_t>(cc >> 1) & 1u) ^ 1u,
                                 status)) {
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
              const uint32_t off = k * Cfg::MMA_K * 4;  // 32 bytes per k step inside the atom
              const uint64_t a_big = smem_desc<Cfg>(st + off);
              const uint64_t a_small = smem_desc<Cfg>(st + Cfg::A_BYTES + off);
              const uint64_t b_big = smem_desc<Cfg>(st + 2 * Cfg::A_BYTES + off);
              const uint64_t b_small = smem_desc<Cfg>(st + 2 * Cfg::A_BYTES + Cfg::B_BYTES + off);
              // The chunk's first MMA overwrites the accumulator (starts the partial sum at 0).
              mma_tf32(acc, a_small, b_big, Cfg::IDESC, (kb != kb0 || k != 0) ? 1u : 0u);
              mma_tf32(acc, a_big, b_small, Cfg::IDESC, 1u);
              mma_tf32(acc, a_big, b_big, Cfg::IDESC, 1u);
            }
            mma_commit(empty(s));  // frees the ring slot when these MMAs are done
          }
          if (ok) mma_commit(accFull + 8u * b);  // the chunk's partial sums are complete
        }
      }
      // Every MMA issued above must finish before TMEM can be released.
      mma_commit(mmaDone);
      mbar_wait_bounded(mmaDone, 0u, status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue: TMEM -> FP32 sums -> C
    const int e = warp - 2;
    const int q = warp & 3;                        // TMEM lanes 32q .. 32q + 31 (rows)
    const int col_base = (e >> 2) * Cfg::EPI_COLS;  // this warp's columns of the tile
    int64_t cc = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
      int m0, n0;
      tile_origin(t, tiles_m, tiles_n, Cfg::BM, Cfg::BN, m0, n0);
      float sum[Cfg::EPI_COLS];
#pragma unroll
      for (int c = 0; c < Cfg::EPI_COLS; ++c) sum[c] = 0.0f;
      for (int kb0 = 0; kb0 < nkb; kb0 += Cfg::CHUNK_KB, ++cc) {
        const int b = static_cast<int>(cc & 1);
        const bool done = !aborted() &&
                          mbar_wait_bounded(accFull + 8u * b, static_cast<uint32_t>(cc >> 1) & 1u, status);
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
        if (lane == 0) mbar_arrive(accEmpty + 8u * b);
      }
      if (!ok) break;
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

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

template <class Cfg>
cudaError_t run_tf32x3(const Problem& p, float* a_big, float* a_small, float* b_big,
                       float* b_small, int64_t Kp) {
  CUtensorMap tAb, tAs, tBb, tBs;
  const CUtensorMapSwizzle sw =
      Cfg::BK == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  cudaError_t e;
  if ((e = encode_tmap_f32_2d(&tAb, a_big, Kp, p.M, Cfg::BK, Cfg::BM, sw)) != cudaSuccess) return e;
  if ((e = encode_tmap_f32_2d(&tAs, a_small, Kp, p.M, Cfg::BK, Cfg::BM, sw)) != cudaSuccess) return e;
  if ((e = encode_tmap_f32_2d(&tBb, b_big, Kp, p.N, Cfg::BK, Cfg::BN, sw)) != cudaSuccess) return e;
  if ((e = encode_tmap_f32_2d(&tBs, b_small, Kp, p.N, Cfg::BK, Cfg::BN, sw)) != cudaSuccess) return e;
  auto kern = tf32x3_kernel<Cfg>;
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
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  const int vec_store = (p.N % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) ? 1 : 0;
  kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, p.stream>>>(
      tAb, tAs, tBb, tBs, p.C, static_cast<int>(p.M), static_cast<int>(p.N),
      static_cast<int>(Kp / Cfg::BK), static_cast<int>(tiles_m), static_cast<int>(tiles_n),
      p.status, vec_store);
  return cudaGetLastError();
}

// Tile widths BN (M is 128): wider tiles read A less often per FLOP; the dispatcher picks
// the width whose tile count spreads evenly over the SMs.
using Tf32N128 = Tf32Config<128, 32, 3, 256>;  // 3 stages of 64 KB, 4 epilogue warps
using Tf32N192 = Tf32Config<192, 16, 4, 256>;  // 4 stages of 40 KB, 8 epilogue warps
using Tf32N224 = Tf32Config<224, 16, 4, 256>;  // 4 stages of 44 KB, 8 epilogue warps
using Tf32N256 = Tf32Config<256, 16, 4, 256>;  // 4 stages of 48 KB, 8 epilogue warps

}  // namespace

// Split planes: A_big, A_small (M x Kp) and B_big, B_small (N x Kp), 4 bytes each, each
// plane starting on a 256-byte boundary.
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int64_t Kp = padded_k(K);
  return 2 * up256(static_cast<size_t>(M) * Kp * 4) + 2 * up256(static_cast<size_t>(N) * Kp * 4);
}

cudaError_t launch_tf32x3(const Problem& p, void* workspace) {
  const int64_t Kp = padded_k(p.K);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t a_plane = up256(static_cast<size_t>(p.M) * Kp * 4);
  const size_t b_plane = up256(static_cast<size_t>(p.N) * Kp * 4);
  float* a_big = reinterpret_cast<float*>(w);
  float* a_small = reinterpret_cast<float*>(w + a_plane);
  float* b_big = reinterpret_cast<float*>(w + 2 * a_plane);
  float* b_small = reinterpret_cast<float*>(w + 2 * a_plane + b_plane);

  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  {
    const int64_t work = p.M * (Kp / 4);
    const int64_t blocks = std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(sms) * 16);
    split_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, p.stream>>>(p.A, a_big, a_small,
                                                                           p.M, p.K, Kp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const int64_t gy = Kp / 32;
    const dim3 grid(static_cast<unsigned>((p.N + 31) / 32),
                    static_cast<unsigned>(gy < 65535 ? gy : 65535));
    split_transpose_kernel<<<grid, dim3(32, 8), 0, p.stream>>>(p.B, b_big, b_small, p.K, p.N, Kp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Persistent CTAs take tiles in rounds of `sms`; the cost of a width is its number of
  // rounds times its width, weighted by the per-tile efficiency measured on GB300 (narrow
  // tiles re-read A more often: 128-wide tiles run about 15 % slower per FLOP than 256).
  const int widths[4] = {128, 192, 224, 256};
  const double weight[4] = {1.15, 1.03, 1.01, 1.0};
  const int64_t tm = (p.M + 127) / 128;
  int best = 0;
  double best_cost = 0.0;
  for (int i = 0; i < 4; ++i) {
    const int64_t tiles = tm * ((p.N + widths[i] - 1) / widths[i]);
    const int64_t rounds = (tiles + sms - 1) / sms;
    const double cost = static_cast<double>(rounds) * widths[i] * weight[i];
    if (i == 0 || cost < best_cost) {
      best = i;
      best_cost = cost;
    }
  }
  if (p.K < 256) best = 0;  // one short chunk: the wide epilogue does not pay
#ifdef TF32X3_FORCE_WIDTH
  best = TF32X3_FORCE_WIDTH;
#endif
  switch (best) {
    case 1: return run_tf32x3<Tf32N192>(p, a_big, a_small, b_big, b_small, Kp);
    case 2: return run_tf32x3<Tf32N224>(p, a_big, a_small, b_big, b_small, Kp);
    case 3: return run_tf32x3<Tf32N256>(p, a_big, a_small, b_big, b_small, Kp);
    default: return run_tf32x3<Tf32N128>(p, a_big, a_small, b_big, b_small, Kp);
  }
}

}  // namespace t2s
