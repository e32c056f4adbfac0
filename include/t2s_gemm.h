/*
 * t2s_gemm.h -- C ABI of the GB300 (sm_103a) FP32 matrix-multiply library.
 *
 * Operation (all entry points): C = A x B in IEEE binary32, row-major, dense
 * (t2s_gemm_bf16_f32 and t2s_gemm_f16_f32 take bfloat16 or binary16 A and B and write a
 * binary32 C; the t2s_gemm_f64 entry points work in binary64 throughout).
 *
 *   A is M x K, element (row, k)   at A[row * K + k]
 *   B is K x N, element (k, col)   at B[k * N + col]
 *   C is M x N, element (row, col) at C[row * N + col]
 *   2 * M * N * K floating-point operations.
 *
 * The layout and index formulas are those of page "GEMM 커널 테스트 코드 작성 및
 * 최적화 (1024^3 크기 실험)", section "메모리 레이아웃"; the per-element operation
 * (one FP32 accumulator per C element, k ascending) is that of its section
 * "Naive GEMM 커널 동작 방식". As on that page, there are no leading dimensions,
 * no alpha/beta scaling and no transposes: the three matrices are dense.
 *
 * Common contract of the GEMM entry points
 * ----------------------------------------
 *  - A, B, C are DEVICE pointers to memory the caller owns (for example from
 *    torch or cudaMalloc) on the current CUDA device. The library keeps no
 *    reference to them after the call returns.
 *  - The call is asynchronous: it validates the arguments on the host,
 *    enqueues kernels on `stream` and returns. `stream` is a cudaStream_t
 *    (NULL = the legacy default stream). Results are visible after the
 *    stream is synchronised.
 *  - A and B must not overlap C (the pages' kernels declare all three
 *    __restrict__). Pointer equality of C with A or B is rejected; partial
 *    overlap is undefined behaviour and not detected.
 *  - Pointers must be 4-byte aligned. No other alignment is required; when
 *    K % 4 == 0, N % 4 == 0 and all three pointers are 16-byte aligned the
 *    product kernel loads tiles with the Tensor Memory Accelerator, otherwise
 *    with 4-byte asynchronous copies. Both give identical results.
 *  - M == 0 or N == 0: nothing to do, returns T2S_OK without touching memory.
 *    K == 0: C is set to +0.0f (the empty sum).
 *  - Each dimension must be <= T2S_MAX_DIM. A pointer may be NULL only if the
 *    matrix it points to has no elements.
 *  - No entry point allocates device or host memory, except that the first
 *    call on a device looks up the address of the library's device status
 *    word (a static device variable; no allocation).
 *
 * Return codes
 *  - T2S_OK:            the kernels were enqueued.
 *  - T2S_ERR_INVALID:   an argument broke the contract; nothing was enqueued.
 *  - T2S_ERR_CUDA:      a CUDA runtime or driver call failed (for example no
 *                       sm_103a device, or a launch error); the CUDA error code
 *                       is available from t2s_last_cuda_error().
 *  - T2S_ERR_WORKSPACE: the workspace passed to t2s_gemm_f32_tf32x3 is NULL
 *                       or smaller than t2s_gemm_f32_tf32x3_workspace_size().
 *  - T2S_ERR_TOO_LARGE: only from t2s_gemm_f32_tf32x3_noalloc: the problem needs
 *                       more scratch than its built-in array holds.
 *  - T2S_ERR_TIMEOUT:   only from t2s_device_status(): a kernel gave up a
 *                       bounded wait on a pipeline barrier (it records this
 *                       in the device status word and returns instead of
 *                       hanging).
 */
#ifndef T2S_GEMM_H
#define T2S_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA header. */
typedef struct CUstream_st *t2s_stream_t;

#define T2S_OK 0
#define T2S_ERR_INVALID 1
#define T2S_ERR_CUDA 2
#define T2S_ERR_TIMEOUT 3
#define T2S_ERR_WORKSPACE 4
#define T2S_ERR_TOO_LARGE 5

#define T2S_MAX_DIM ((int64_t)1 << 30) /* per dimension */

/*
 * The product kernel. FP32 fused multiply-adds on the CUDA cores (packed
 * two-wide, one rounding each), one accumulator per C element summed in
 * ascending k, CTA tiles staged through shared memory by a multi-stage
 * barrier pipeline. Because every step is an IEEE fused multiply-add taken in
 * the page's order, the result is bit-identical to the definition evaluated
 * with fmaf() (page "GEMM 커널 테스트 코드 작성 및 최적화 (1024^3 크기 실험)",
 * section "Naive GEMM 커널 동작 방식" read with nvcc's default contraction), for
 * every input. The tiling follows page "4주차: Roofline과 Tiling", section
 * "3. Tiling": each tile of A and B is read from HBM once per CTA tile and
 * reused from shared memory and registers.
 */
int t2s_gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                 float *C, t2s_stream_t stream);

/*
 * The CTA tiling t2s_gemm_f32 takes for an M x N x K product on a GPU with `sms`
 * multiprocessors (page "4주차: Roofline과 Tiling", item 8 of "이번 주차 핵심": the tile is
 * chosen per problem, large tiles for reuse, small ones to fill the machine). A host-only
 * query: it touches no device, and every choice gives the same bits.
 *  - Returns 0: 128 x 128 tiles, k loop unrolled over a K block; 1: 128 x 128 tiles, compact
 *    k loop; 2: 128 x 64 tiles; 3: 64 x 64 tiles; 4: 256 x 128 tiles; 5: 256 x 128 tiles in
 *    whole rounds of `sms` tiles, then the remaining 256 x 128 tiles as 64 x 64 tiles in a
 *    second launch; 6: 128 x 128 tiles of 8 warps; 7: 128 x 64 tiles of 8 warps (6 and 7 only
 *    for at most one tile per multiprocessor); 9: 56 x 128 tiles of 8 warps (at most one per
 *    multiprocessor, or from K = 128 on also more, two CTAs sharing each); 8: 128 x 128
 *    tiles on a persistent grid of two CTAs per multiprocessor, one TMA ring across tiles
 *    (K <= 32; on the cp.async path the call runs 1 instead); 10: 32 x 32 tiles (small
 *    products); 11: 256 x 128 tiles on a persistent grid of one CTA per multiprocessor whose
 *    warps hand C to TMA stores while they go on to the next tile (K <= 96 and at least two
 *    rounds of such tiles; on the cp.async path, or when C is not 16-byte aligned, the call
 *    runs 1 instead). -1 if a dimension is negative or above T2S_MAX_DIM, or sms < 1.
 */
int t2s_gemm_f32_plan(int64_t M, int64_t N, int64_t K, int sms);

/*
 * The product of t2s_gemm_f32 for matrices in HOST memory (row-major, same layout),
 * staged through device buffers the caller owns: dA (M*K floats), dB (K*N), dC (M*N).
 * Copies run on their own streams under the products, in one of two schedules, whichever
 * leaves fewer bytes to copy before the first product starts:
 *  - row blocks: copy B, then stream A in row blocks, multiplying each block as soon as it
 *    has arrived and copying its block of C back while later blocks compute;
 *  - K chunks (K of at least two chunks of about 1024): stream A and B in chunks of K
 *    (columns of A, rows of B); the product over each chunk resumes from the partial sums
 *    the previous chunk stored in dC, and the last chunk runs in row blocks whose blocks of
 *    C are copied back as they finish.
 * Either way every element is the same chain of fused multiply-adds in ascending k, so the
 * result is bit-identical to t2s_gemm_f32.
 *  - hA, hB, hC should be page-locked (cudaHostAlloc, cudaHostRegister) for the copies to
 *    run asynchronously and overlap; pageable memory gives the same result, serialised.
 *  - Asynchronous: returns once everything is enqueued; hC is complete, and hA, hB, dA,
 *    dB, dC may be reused, after `stream` has been synchronised.
 *  - Allocates no device memory. The first call on a device creates three streams and
 *    twenty-one events that the library keeps for later calls; calls from several host
 *    threads are serialised while they enqueue.
 *  - Errors: T2S_ERR_INVALID as for t2s_gemm_f32 (a NULL buffer for a non-empty matrix,
 *    dC equal to dA or dB); T2S_ERR_CUDA if a copy, event or launch fails.
 */
int t2s_gemm_f32_host(int64_t M, int64_t N, int64_t K, const float *hA, const float *hB,
                      float *hC, float *dA, float *dB, float *dC, t2s_stream_t stream);

/*
 * Comparison point: one thread per C element, k loop over global memory,
 * 16 x 16 thread blocks (page "GEMM 커널 테스트 코드 작성 및 최적화 (1024^3 크기
 * 실험)", sections "Naive GEMM 커널 동작 방식" and "쓰레드 매핑"). Uses fmaf, so
 * its result is bit-identical to t2s_gemm_f32.
 */
int t2s_gemm_f32_naive(int64_t M, int64_t N, int64_t K, const float *A,
                       const float *B, float *C, t2s_stream_t stream);

/*
 * Comparison point: 32 x 32 shared-memory tiles, one C element per thread,
 * zero-filled ragged edges, two block barriers per K tile (same page, sections
 * "Shared Memory Tiled GEMM 연산 방식", "타일 개념", "타일 로딩 단계"). Uses
 * fmaf, so its result is bit-identical to t2s_gemm_f32.
 */
int t2s_gemm_f32_smem32(int64_t M, int64_t N, int64_t K, const float *A,
                        const float *B, float *C, t2s_stream_t stream);

/*
 * Split-K product for small or short-K problems (item "split-K for small and low-K shapes"
 * of the tiling plan; page "4주차: Roofline과 Tiling", item 8 of "이번 주차 핵심": tiles that
 * are too large for the problem leave the machine idle). K is cut into `splits` chunks of
 * ceil(K / splits) values rounded up to 32; each chunk's product is computed by the product
 * kernel into its own plane of `workspace` (M x N floats per plane), and the planes are then
 * added into C in chunk order. Each chunk is summed in ascending k with fused multiply-adds,
 * so the result differs from t2s_gemm_f32 only by the order of the chunk sums: it is
 * deterministic and within max |C - C_fp32| <= 1e-6 * K * max|a| * max|b|, but not
 * bit-identical.
 *  - splits: 1..64 chunks requested, or <= 0 for the library's choice: the count from 1 (no
 *    split) to 16, chunks of at least 128 values, whose modelled time is least. The model is
 *    the busiest SM's work under the product's own tiling choice, plus the bytes of the plane
 *    sum. With a single chunk the call is t2s_gemm_f32.
 *  - workspace: a DEVICE buffer, 256-byte aligned, of at least
 *    t2s_gemm_f32_splitk_workspace_size(M, N, K, splits) bytes (0 if no split is made), owned
 *    by the caller and untouched until the stream has run the call.
 *  - Returns T2S_ERR_INVALID for splits > 64, T2S_ERR_WORKSPACE for a missing, small or
 *    misaligned workspace, otherwise as t2s_gemm_f32.
 */
size_t t2s_gemm_f32_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int splits);

/*
 * The chunk count t2s_gemm_f32_splitk takes for splits <= 0 on a GPU with `sms`
 * multiprocessors (1 means no split: the call is t2s_gemm_f32). A host-only query: it
 * touches no device. -1 if a dimension is negative or above T2S_MAX_DIM, or sms < 1.
 */
int t2s_gemm_f32_splitk_plan(int64_t M, int64_t N, int64_t K, int sms);
int t2s_gemm_f32_splitk(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                        float *C, int splits, void *workspace, size_t workspace_bytes,
                        t2s_stream_t stream);

/*
 * Stream-K product for shapes whose tiles do not divide evenly over the GPU (small and mid
 * sizes; the last partial wave of large ones). The iterations of the product -- 128 x 128
 * tiles times 32-deep K blocks, tiles in the product kernel's order, K blocks ascending --
 * are shared out in equal contiguous ranges over a persistent grid of two CTAs per SM, so
 * every SM gets the same work whatever the tile count. A tile whose K blocks all fall in one
 * CTA's range is stored into C by that CTA; the CTAs that share a tile store their partial
 * sums of it in `workspace`, and a second kernel adds those partial tiles in K order. The
 * result is deterministic and within max |C - C_fp32| <= 1e-6 * K * max|a| * max|b|, but not
 * bit-identical to t2s_gemm_f32 (a shared tile's partial sums are added at the end).
 *  - workspace: a DEVICE buffer, 256-byte aligned, of at least
 *    t2s_gemm_f32_streamk_workspace_size(M, N, K) bytes (two 128 x 128 float tiles per CTA,
 *    about 40 MB on a 152-SM GB300), owned by the caller and untouched until the stream has
 *    run the call; T2S_ERR_WORKSPACE if NULL, too small or misaligned.
 *  - Needs the TMA path (K % 4 == 0, N % 4 == 0, A and B 16-byte aligned); other shapes run
 *    the product kernel (bit-identical to t2s_gemm_f32) and leave the workspace unused.
 *  - Otherwise the common contract and return codes above apply.
 */
size_t t2s_gemm_f32_streamk_workspace_size(int64_t M, int64_t N, int64_t K);
int t2s_gemm_f32_streamk(int64_t M, int64_t N, int64_t K, const float *A, const float *B,
                         float *C, void *workspace, size_t workspace_bytes,
                         t2s_stream_t stream);

/*
 * Tensor-core variant: error-compensated 3xTF32 on tcgen05 tensor cores with
 * TMEM accumulators. Each operand x is split into big = tf32(x) and
 * small = tf32(x - big); C accumulates small*big + big*small + big*big in FP32.
 * This is not on the pages (the split is from Ootomo and Yokota, "Recovering
 * single precision accuracy from Tensor Cores while surpassing the FP32
 * theoretical peak performance", 2022). The result is not bit-identical to the
 * FP32 definition (the tensor core fixes its own summation order); it meets
 * max |C - C_fp32| <= 1e-6 * K * max|a| * max|b|, and it is exact wherever
 * every FP32 product and partial sum is exact (for example small integers).
 * A NaN operand gives NaN where the definition does; an infinite operand may give
 * NaN where the definition gives an infinity (a correction term multiplies it by
 * the zero small part of an operand that TF32 represents exactly). Finite operands
 * stay finite in the split, up to FLT_MAX: a value within half a TF32 ulp of it,
 * which would round up to infinity, keeps its truncated TF32 value as big and the
 * exact remainder goes into small, so results that are finite in the definition
 * stay finite and within the bound.
 *
 * `workspace` is a DEVICE buffer, 256-byte aligned, of at least
 * t2s_gemm_f32_tf32x3_workspace_size(M, N, K) bytes, owned by the caller,
 * that holds the split operands; it must not overlap A, B or C and must stay
 * untouched until the stream has run the call. Returns T2S_ERR_WORKSPACE if it
 * is NULL, too small or not 256-byte aligned.
 */
size_t t2s_gemm_f32_tf32x3_workspace_size(int64_t M, int64_t N, int64_t K);
int t2s_gemm_f32_tf32x3(int64_t M, int64_t N, int64_t K, const float *A,
                        const float *B, float *C, void *workspace,
                        size_t workspace_bytes, t2s_stream_t stream);

/*
 * The same 3xTF32 product for callers that cannot allocate device memory (the source
 * pages have no counterpart of this entry point). Examples: a plugin inside a framework
 * that owns all device memory through its own pool and budget, a latency-critical loop
 * that cannot afford the implicit synchronisation and unbounded time of cudaMalloc /
 * cudaFree, or C code without a device allocator of its own.
 *
 * Instead of a caller-owned workspace, the split operands live in a static device array of
 * T2S_TF32X3_NOALLOC_MAX_SCRATCH bytes (32 MiB) inside this library. Every GPU that loads
 * the library holds that array until the process exits. The call allocates nothing and
 * calls no allocating routine.
 *  - Limit: t2s_gemm_f32_tf32x3_workspace_size(M, N, K), which is about
 *    8 * (M + N) * ceil(K / 32) * 32 bytes (four planes of 4-byte values), must not exceed
 *    T2S_TF32X3_NOALLOC_MAX_SCRATCH. M = N = K = 1024 takes 16 MiB; the largest square
 *    product that fits is 1440^3. Larger problems return T2S_ERR_TOO_LARGE and enqueue
 *    nothing.
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *    once per device); make that first call before any stream capture begins.
 *  - All calls on a device share the one array, which keeps the last call's contents. Each
 *    call rewrites every byte it reads, so nothing needs clearing between calls. Calls
 *    that can overlap on the GPU (for example on two streams without ordering between
 *    them) race on the array and may return wrong results: order them.
 *  - Otherwise the contract, results and return codes are those of t2s_gemm_f32_tf32x3.
 */
#define T2S_TF32X3_NOALLOC_MAX_SCRATCH ((size_t)32 << 20)
int t2s_gemm_f32_tf32x3_noalloc(int64_t M, int64_t N, int64_t K, const float *A,
                                const float *B, float *C, t2s_stream_t stream);

/*
 * BF16 element type on the tcgen05 tensor cores: C (FP32) = A x B with A and B in bfloat16.
 * The pages write their kernels for a template element type T (page "GEMM 커널 테스트 코드
 * 작성 및 최적화 (1024^3 크기 실험)", sections "Naive GEMM 커널 동작 방식" and "Shared
 * Memory Tiled GEMM 연산 방식"); this is the 16-bit instance on GB300's tensor cores, with FP32
 * accumulation (tcgen05.mma kind::f16, BF16 operands).
 *
 * Layout: A is M x K and B is K x N, row-major, dense, as uint16_t bit patterns of IEEE-style
 * bfloat16 (the upper 16 bits of a binary32); C is M x N row-major FP32. Every product of two
 * bfloat16 values is exact in FP32, so C differs from the FP32 definition applied to the
 * bfloat16 values only in the order of the FP32 additions: exact wherever all products and
 * partial sums are (for example small integers); otherwise
 * max |C - sum_k a*b| <= 1e-6 * K * max|a| * max|b|.
 *
 * A and B must be 2-byte aligned, C 4-byte aligned. When K % 8 == 0 and A is 16-byte aligned,
 * A is read in place; otherwise it is first copied into a padded plane of the workspace.
 * `workspace` is a DEVICE buffer, 256-byte aligned, of at least
 * t2s_gemm_bf16_f32_workspace_size(M, N, K) bytes, owned by the caller, holding B transposed
 * (and A padded); it must not overlap A, B or C and must stay untouched until the stream has
 * run the call. Otherwise the common contract and return codes above apply.
 */
size_t t2s_gemm_bf16_f32_workspace_size(int64_t M, int64_t N, int64_t K);
int t2s_gemm_bf16_f32(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                      float *C, void *workspace, size_t workspace_bytes, t2s_stream_t stream);

/*
 * The same product for IEEE 754 binary16 (FP16) A and B: uint16_t bit patterns with 1 sign,
 * 5 exponent (bias 15) and 10 fraction bits, subnormals included. Every product of two FP16
 * values is exact in FP32, so the same bars hold: exact wherever every partial sum is exact,
 * otherwise max |C - sum_k a*b| <= 1e-6 * K * max|a| * max|b|. Layout, alignment, workspace
 * (the same size as for BF16), contract and return codes are those of t2s_gemm_bf16_f32.
 */
size_t t2s_gemm_f16_f32_workspace_size(int64_t M, int64_t N, int64_t K);
int t2s_gemm_f16_f32(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B,
                     float *C, void *workspace, size_t workspace_bytes, t2s_stream_t stream);

/*
 * FP64 element type on the CUDA cores: C = A x B in IEEE binary64, the same layout and
 * definition as the FP32 entry points with T = double (page "GEMM 커널 테스트 코드 작성 및
 * 최적화 (1024^3 크기 실험)": both kernels there are templates over the element type).
 *  - t2s_gemm_f64: the product; 32 x 32 CTA tiles staged through shared memory in 16-deep K
 *    tiles, 2 x 2 register blocks per thread (page "4주차: Roofline과 Tiling", section
 *    "3. Tiling"), sized for balance across the SMs: GB300's FP64 rate (2 FMA per SM per
 *    clock) is reached at any tiling.
 *  - t2s_gemm_f64_naive: one thread per C element, k loop over global memory, 16 x 16 blocks.
 *  - t2s_gemm_f64_smem32: 32 x 32 shared-memory tiles, one C element per thread.
 * All three sum each element with one IEEE fused multiply-add (fma) per k in ascending k, so
 * they are bit-identical to each other and to the definition evaluated with fma(), for every
 * input. Pointers must be 8-byte aligned; otherwise the common contract and return codes
 * above apply (K == 0 sets C to +0.0).
 */
int t2s_gemm_f64(int64_t M, int64_t N, int64_t K, const double *A, const double *B,
                 double *C, t2s_stream_t stream);
int t2s_gemm_f64_naive(int64_t M, int64_t N, int64_t K, const double *A, const double *B,
                       double *C, t2s_stream_t stream);
int t2s_gemm_f64_smem32(int64_t M, int64_t N, int64_t K, const double *A, const double *B,
                        double *C, t2s_stream_t stream);

/*
 * Memory-roof probe: z[i] = x[i] + y[i] for i < n, FP32, one IEEE add (round to nearest)
 * per element. This is the memory-bound example of page "4주차: Roofline과 Tiling", section
 * "1. Arithmetic Intensity" ("Vector Add": N FLOPs for 12N bytes moved, AI = 1/12 FLOP/B);
 * its measured bandwidth is the slope of the roofline on which the GEMM kernels are placed.
 * x, y, z are device pointers (4-byte aligned; 32-byte alignment of all three selects the
 * widest loads); z must not overlap x or y (exact aliasing is rejected). Asynchronous on
 * `stream`; n == 0 is a no-op. Returns T2S_OK, T2S_ERR_INVALID or T2S_ERR_CUDA.
 */
int t2s_vector_add_f32(int64_t n, const float *x, const float *y, float *z,
                       t2s_stream_t stream);

/* Static description of a return code. Never NULL. */
const char *t2s_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the status word of the current
 * device. Returns T2S_OK, T2S_ERR_TIMEOUT if a kernel since the last read gave
 * up a bounded barrier wait, or T2S_ERR_CUDA if synchronising or reading failed.
 */
int t2s_device_status(t2s_stream_t stream);

/* The last CUDA error code seen by a failing call on this host thread (0 if none). */
int t2s_last_cuda_error(void);

/*
 * Self-test of the bounded-wait mechanism: launches one block that waits on a
 * barrier nothing will ever complete, with a limit of `limit_ns` nanoseconds
 * (clamped to [1e3, 1e9]). The kernel records T2S_ERR_TIMEOUT in the status
 * word and returns; t2s_device_status() then reports it. Returns T2S_OK if
 * the kernel was enqueued.
 */
int t2s_selftest_wait_timeout(int64_t limit_ns, t2s_stream_t stream);

/*
 * Throughput probes: the measured ceilings of the roofline (page "4주차: Roofline과 Tiling",
 * section "2. Roofline": a kernel's attainable performance is min(peak FLOP/s, bandwidth x
 * arithmetic intensity); the pages give no GB300 peaks, so they are measured). Each launches
 * one kernel on `stream` and stores in *flops (host memory) the floating-point operations it
 * performs; the caller times the launch (CUDA events on `stream`) and divides.
 *  - t2s_probe_fp32_fma: every thread of 2 CTAs of 128 threads per SM (the product kernels'
 *    8 warps per SM) runs `iters` rounds of 16 independent packed fused multiply-adds
 *    (fma.rn.f32x2, 4 FLOP each) with no memory traffic. iters in [1, 2^24].
 *  - t2s_probe_tf32_mma: one CTA per SM issues `iters` x 4 back-to-back tcgen05.mma
 *    kind::tf32 of M = 128, N = 256, K = 8 (2 x 128 x 256 x 8 FLOP each) on operands resident
 *    in shared memory, accumulating in TMEM: the instruction and operand layout of the 3xTF32
 *    product. iters in [1, 2^16]; the wait for the MMAs is bounded (T2S_ERR_TIMEOUT through
 *    t2s_device_status).
 * `out` is a DEVICE buffer of at least t2s_probe_outputs() floats (one value per thread,
 * written so that the work is observable). Returns T2S_OK, T2S_ERR_INVALID (iters out of
 * range, NULL pointer) or T2S_ERR_CUDA.
 */
int t2s_probe_outputs(void);
int t2s_probe_fp32_fma(int64_t iters, float *out, int64_t *flops, t2s_stream_t stream);
int t2s_probe_tf32_mma(int64_t iters, float *out, int64_t *flops, t2s_stream_t stream);

/*
 * Store-path probe: the rate at which a matrix leaves the SMs, the ceiling of every product
 * whose C is as large as its arithmetic (short K). Writes `value` to every element of the
 * row-major M x N FP32 matrix C with no arithmetic, in the short-K product's store pattern:
 * one CTA of 8 warps per SM walks 256 x 128 tiles in the product's grouped order (groups of 8
 * tile rows), each warp writing a 64 x 64 part, either
 *  - mode 0: staged in shared memory and stored as two 64 x 32 TMA boxes (128-byte swizzle),
 *    restaged once the previous stores have read the boxes (the short-K kernel's epilogue), or
 *  - mode 1: as 16-byte stores from registers in the register-tile layout (the epilogue of
 *    the other product kernels).
 * C is a DEVICE pointer, 16-byte aligned; M a multiple of 256 and N a multiple of 128, both
 * positive and at most T2S_MAX_DIM. *bytes (host memory) receives the bytes written, 4 M N;
 * the caller times the launch on `stream`. Returns T2S_OK, T2S_ERR_INVALID (sizes, alignment,
 * mode, NULL pointers; checked before any device call) or T2S_ERR_CUDA.
 */
int t2s_probe_store_f32(int64_t M, int64_t N, float *C, int mode, float value, int64_t *bytes,
                        t2s_stream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int t2s_version(void);

#ifdef __cplusplus
}
#endif

#endif /* T2S_GEMM_H */
