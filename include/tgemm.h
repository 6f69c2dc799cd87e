/*
 * tgemm: tiled dense matrix multiply C = A * B for one NVIDIA GB300 (sm_103a).
 *
 * The operation is the defining sum of "Writing high-performance matrix
 * multiplication with NVIDIA CUDA Tile" (juejin.cn, section "What is matrix
 * multiplication?"):  C[i][j] = sum_k A[i][k] * B[k][j],  with the precision
 * contract of the CUDA Programming Guide 13.4.2 (unofficial Chinese
 * translation), section 2.4.9.1 "Matrix multiplication": FP16 or BF16
 * operands, an FP32 accumulator, one cast to the output type at the store.
 * Tails follow the same section: the K loop runs ceil(K / tile_k) times with
 * the partial K tile zero-padded, and partial M/N edge tiles drop their
 * out-of-range elements at the store.
 *
 * Conventions shared by every entry point:
 *   - All matrices are row-major.  A is M x K: A[i*lda + k].  C is M x N:
 *     C[i*ldc + j].  B is K x N stored either as B[k*ldb + j]
 *     (TGEMM_B_KN) or as its transpose, N x K: B[j*ldb + k] (TGEMM_B_NK).
 *   - Leading dimensions are in elements.  ld * element size must be a
 *     multiple of 16 bytes and every base pointer 16-byte aligned (the tensor
 *     memory accelerator addresses rows in 16-byte units; CUDA Programming
 *     Guide 13.4.2, section 2.4.12.2 "Mark array pointers as 16-byte
 *     aligned").  There is no unaligned fallback.
 *   - A, B and C are device memory owned by the caller and must not overlap
 *     (section 2.4.12.1 of the same guide: __restrict__ arrays).  C is
 *     overwritten, never accumulated into.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream).  Argument errors are detected on the host
 *     before anything is launched and leave C untouched.
 *   - The library owns only a 4-byte device status word per device, its
 *     split-K workspace and a host cache of tensor descriptors; all are freed
 *     by tgemm_shutdown().  Entry points are thread-safe.
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { TGEMM_B_KN = 0, TGEMM_B_NK = 1 } tgemm_b_layout;

/* Element types.  FP8 (E4M3 "fn" variant with no infinities, E5M2) is an
 * input type only: both operands the same FP8 type, B stored N x K, FP32
 * accumulation, FP16/BF16/FP32 output (scale factors go in the epilogue's
 * alpha).  TGEMM_F32 as in_dtype means FP32 operands multiplied on the
 * tensor cores as TF32: each element's low 13 fraction bits are dropped
 * (truncation toward zero, as the tensor core reads 32-bit containers), the
 * products are summed in FP32; B stored N x K.  The cuTile tutorial gives
 * FP32 operands their own tile shape ("Launching the kernel from the host")
 * without saying how they are multiplied. */
typedef enum { TGEMM_F16 = 0, TGEMM_BF16 = 1, TGEMM_F32 = 2, TGEMM_E4M3 = 3, TGEMM_E5M2 = 4 } tgemm_dtype;

typedef enum {
    TGEMM_OK = 0,
    TGEMM_ERR_INVALID_ARG = 1,   /* negative size, NULL pointer, ld shorter than a row, bad enum  */
    TGEMM_ERR_UNSUPPORTED = 2,   /* dtype combination or configuration the kernels do not provide */
    TGEMM_ERR_MISALIGNED = 3,    /* pointer not 16-byte aligned or ld*elem not a multiple of 16   */
    TGEMM_ERR_ARCH = 4,          /* current device is not compute capability 10.3 (sm_103)         */
    TGEMM_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed                               */
    TGEMM_ERR_OOM = 6,           /* library-owned workspace could not be allocated                 */
    TGEMM_ERR_TIMEOUT = 7        /* a kernel gave up on a pipeline wait and recorded it (see check) */
} tgemm_status;

/*
 * A kernel configuration.  bm x bn is the output tile of one CTA pair
 * (cluster_m = 2) or one CTA (cluster_m = 1); bk is the K depth of one
 * pipeline stage; stages is the shared-memory ring depth; group_m is the
 * GROUP_SIZE_M of the grouped rasterisation ("Performance optimisation:
 * Swizzle" of the cuTile matrix multiplication tutorial); swap_ab != 0
 * computes C^T = B^T A^T so a short M (padded to bn) becomes the MMA's N,
 * with the K loop split over split_k CTAs whose partial sums are added
 * through a global FP32 workspace (swap_ab = 1: M <= 64, bn 16/32/64) or
 * inside a thread-block cluster of split_k CTAs (swap_ab = 2, cluster_m =
 * split_k: M <= 128, bn 16/32/64/128, at most 4 splits for 128; FP16/BF16
 * and FP8 operands, the workspace form FP16/BF16 only); grid is the number
 * of CTAs launched (0 = the library's choice).  Tile kernels: cluster_m = 1
 * (bm 128, bn 128 or 256; bn 128 also with stages = 2, two CTAs per SM,
 * FP16/BF16 only), 2 (a CTA pair, 256 x 256) or 4
 * (two CTA pairs on neighbouring 256 x 256 tiles sharing their A rows); for
 * cluster_m = 2 and 4, split_k = 0 adds a stream-K tail (the last waves'
 * tiles, or the quad's 256 x 512 blocks, shared out by k-range and summed
 * in a fixed order).
 */
typedef struct {
    int bm, bn, bk, stages, cluster_m, group_m, split_k, swap_ab, grid;
} tgemm_config;

/*
 * C = A * B.  in_dtype (TGEMM_F16, TGEMM_BF16, TGEMM_E4M3, TGEMM_E5M2 or
 * TGEMM_F32, see tgemm_dtype) is the type of both A and B; out_dtype is
 * TGEMM_F16, TGEMM_BF16 or TGEMM_F32.  FP8 and FP32 operands need B stored
 * N x K (TGEMM_B_NK), else TGEMM_ERR_UNSUPPORTED.  M, N or K may be 0:
 * M = 0 or N = 0 is a no-op; K = 0 writes zeros (the empty sum).
 * Returns TGEMM_OK once the work is enqueued on `stream`.
 */
tgemm_status tgemm_run(int64_t M, int64_t N, int64_t K,
                       const void *A, int64_t lda,
                       const void *B, int64_t ldb, tgemm_b_layout b_layout,
                       void *C, int64_t ldc,
                       tgemm_dtype in_dtype, tgemm_dtype out_dtype, void *stream);

/*
 * Fused epilogue: D = act(alpha * (A * B) + beta * C_in + bias), evaluated
 * in FP32 on the accumulator and cast once to out_dtype.  The Croqtile
 * tutorial counts epilogue fusion among cuBLAS's advantages (its comparison
 * with cuBLAS); this is the usual affine-plus-activation form.
 *   alpha    scale of the product (1 = none)
 *   beta     scale of C_in; 0 = C_in is not read
 *   c_in     M x N matrix of type out_dtype, row pitch ldc_in (elements); may be
 *            C itself (in-place accumulate); 16-byte aligned like C
 *   bias     N values of type bias_dtype added to every row, or NULL; 16-byte
 *            aligned
 *   act      TGEMM_ACT_NONE, TGEMM_ACT_RELU (max(x, 0)) or TGEMM_ACT_GELU_TANH
 *            (0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))))
 */
typedef enum { TGEMM_ACT_NONE = 0, TGEMM_ACT_RELU = 1, TGEMM_ACT_GELU_TANH = 2 } tgemm_activation;

typedef struct {
    float alpha;
    float beta;
    const void *c_in;
    int64_t ldc_in;
    const void *bias;
    tgemm_dtype bias_dtype;
    tgemm_activation act;
} tgemm_epilogue;

/* tgemm_run with a fused epilogue (ep may be NULL: plain C = A * B) and an
 * optional explicit configuration (cfg NULL: the library's choice).  With
 * K = 0 the product is the empty sum and D = act(beta * C_in + bias). */
tgemm_status tgemm_run_ex(int64_t M, int64_t N, int64_t K,
                          const void *A, int64_t lda,
                          const void *B, int64_t ldb, tgemm_b_layout b_layout,
                          void *C, int64_t ldc,
                          tgemm_dtype in_dtype, tgemm_dtype out_dtype, void *stream,
                          const tgemm_epilogue *ep, const tgemm_config *cfg);

/*
 * `batch` independent products C_b = A_b * B_b (b = 0 .. batch-1), the batched
 * form of the CUDA Programming Guide 13.4.2 (unofficial Chinese translation),
 * section 2.4.9.1 ("matmul and mma support 3-D batched multiplication"):
 * A_b at A + b*stride_a, B_b at B + b*stride_b, C_b at C + b*stride_c
 * (strides in elements).  A stride of 0 shares that operand across every
 * batch; otherwise strides must not make batches overlap (stride_a >= M*lda,
 * stride_b >= rows*ldb, stride_c >= M*ldc) and must keep 16-byte alignment.
 * With an epilogue, C_in steps like C.  All batches run in one launch of the
 * tile kernels (the skinny-M kernels are not batched).  batch = 0 is a no-op.
 */
tgemm_status tgemm_run_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                                       const void *A, int64_t lda, int64_t stride_a,
                                       const void *B, int64_t ldb, int64_t stride_b, tgemm_b_layout b_layout,
                                       void *C, int64_t ldc, int64_t stride_c,
                                       tgemm_dtype in_dtype, tgemm_dtype out_dtype, void *stream,
                                       const tgemm_epilogue *ep, const tgemm_config *cfg);

/* The configuration tgemm_run would use for this problem (no device work,
 * but it reads the current device's SM count and compute capability).  The
 * pages leave tile sizes to the launcher ("Launching the kernel from the
 * host" of the cuTile matrix multiplication tutorial picks them per dtype)
 * and to measurement ("CUDA 13.1 new feature: the Tile programming model",
 * section 7, autotuning over tile shapes); this returns the per-shape choice
 * that the library's measured table or, off its grid, its wave model makes.
 * With TGEMM_LOG set (not "0") every GEMM entry point prints the
 * configuration it launched, one line per call on stderr. */
tgemm_status tgemm_query_config(int64_t M, int64_t N, int64_t K, tgemm_b_layout b_layout,
                                tgemm_dtype in_dtype, tgemm_dtype out_dtype,
                                tgemm_config *out_cfg);

/* tgemm_query_config for a GPU with `sm_count` SMs given by the caller
 * (1..4096), touching no device: for planning and host-side tests.  The
 * choice assumes tightly packed rows (lda = K; ldb = K for TGEMM_B_NK, N for
 * TGEMM_B_KN), as tgemm_query_config does; with the current device's SM
 * count the two return the same configuration.  Returns
 * TGEMM_ERR_INVALID_ARG or TGEMM_ERR_UNSUPPORTED for the arguments
 * tgemm_query_config rejects, and TGEMM_ERR_INVALID_ARG for an SM count
 * outside that range. */
tgemm_status tgemm_query_config_sms(int64_t M, int64_t N, int64_t K, tgemm_b_layout b_layout,
                                    tgemm_dtype in_dtype, tgemm_dtype out_dtype, int sm_count,
                                    tgemm_config *out_cfg);

/* tgemm_run with an explicit configuration, for tuning and tests: the
 * measurement side of the autotuning the pages describe (the Tile
 * programming model overview, section 7, times candidate tile shapes; the
 * cuTile tutorial's launcher fixes them by hand).  A configuration the
 * kernels do not provide returns TGEMM_ERR_UNSUPPORTED. */
tgemm_status tgemm_run_config(int64_t M, int64_t N, int64_t K,
                              const void *A, int64_t lda,
                              const void *B, int64_t ldb, tgemm_b_layout b_layout,
                              void *C, int64_t ldc,
                              tgemm_dtype in_dtype, tgemm_dtype out_dtype, void *stream,
                              const tgemm_config *cfg);

/* Synchronise `stream`, then report the first failure since the last check:
 * a pending CUDA error (TGEMM_ERR_CUDA) or a kernel that timed out on a
 * pipeline wait (TGEMM_ERR_TIMEOUT; the status word is then cleared).  Both
 * the library's status word and the allocation-free entry point's are read.
 * The Croqtile tutorial's summary warns that a hand-written warp-specialised
 * pipeline can deadlock silently; every wait here is bounded instead, and
 * this call is where a wait that gave up becomes visible to the caller. */
tgemm_status tgemm_check(void *stream);

/* The last non-zero status word tgemm_check read (0 = none): bits 28-31 the
 * fault class (7 = timeout), bits 20-27 the wait site, bits 0-19 the CTA;
 * for diagnostics after tgemm_check (the same silent-deadlock passage). */
uint32_t tgemm_last_fault_code(void);

/* A short English description of a status code (never NULL).  The codes are
 * the boundary's failure classes: argument checks from the CUDA Programming
 * Guide 13.4.2 (unofficial Chinese translation), sections 2.4.12.1-2.4.12.2
 * (non-overlapping __restrict__ arrays, 16-byte aligned rows), the GB300
 * architecture check, CUDA errors, workspace allocation and the bounded-wait
 * timeout. */
const char *tgemm_status_string(tgemm_status s);

/* Free every library-owned resource on every device it touched: the status
 * words, the split-K / stream-K workspaces and the tensor-descriptor cache.
 * The pages' kernels own no memory beyond their operands (the cuTile
 * tutorial's launcher allocates only C); this state exists because the
 * persistent kernels here share tail tiles by k-range (the Croqtile
 * tutorial's comparison with cuBLAS names persistent kernels as its edge),
 * so this call has no counterpart on the pages.  The allocation-free entry
 * point's built-in array is not freed: it lives as long as the library. */
void tgemm_shutdown(void);

/*
 * The grouped tile rasterisation used by the persistent scheduler, exposed
 * for host-side tests: tile number `bid` of a grid of ceil(M/bm) x ceil(N/bn)
 * output tiles maps to (tile row *bid_m, tile column *bid_n).  This is the
 * swizzle_2d_from_bid mapping of "Writing high-performance matrix
 * multiplication with NVIDIA CUDA Tile", section "Performance optimisation:
 * Swizzle".  Returns TGEMM_ERR_INVALID_ARG if bid is outside the grid.
 */
tgemm_status tgemm_tile_coord(int64_t M, int64_t N, int bm, int bn, int group_m, int64_t bid,
                              int64_t *bid_m, int64_t *bid_n);

/*
 * The group_m (bands of tile rows of the grouped order above) that an L2
 * footprint model gives for a single problem on the tile kernels, exposed
 * for host-side tests; no device is touched.  tgemm_run and
 * tgemm_query_config use it in place of a default group of 8 when it is
 * taller; a group the picker table measured stays.  bm x unit_bn is the
 * unit the order deals out (a tile, or a quad's 256 x 512 block) and
 * `resident` how many units run at once.  The tutorial's group of 8 is kept
 * while A and B together fit in 96 MiB of L2 or a band of 8 rows holds fewer
 * than two waves of units; otherwise the fewest bands of near-equal height
 * whose A rows, two waves' B columns and one wave's C fit in 64 MiB, or the
 * band with the smallest such footprint.  That section of the tutorial
 * explains the order by L2 reuse; the sizes are this library's.  Returns
 * TGEMM_ERR_INVALID_ARG for a size below 1, an unknown dtype or a NULL
 * output.
 */
tgemm_status tgemm_group_size(int64_t M, int64_t N, int64_t K, int bm, int unit_bn, int in_dtype, int out_dtype,
                              int resident, int *group_m);

/*
 * The stream-K plan of a pair (tiles_per_item = 1) or quad (2: its 256 x 512
 * blocks) launch, exposed for host-side tests; no device is touched.  `items`
 * work items of `k_blocks` k-blocks each run on `units` resident CTA pairs or
 * quads.  On return the first *dp_items items are dealt out whole and the
 * *sk_items after them are shared by *sk_units units, unit u taking k-block
 * iterations [u * I / U, (u + 1) * I / U) of the I = sk_items * k_blocks
 * shared ones, U = *sk_units (floor division).  *sk_units = 0 (with
 * *dp_items = items) keeps every item whole.  Sharing splits work by
 * iterations instead of tiles, a choice of this library: the pages deal
 * whole tiles to blocks.  Returns TGEMM_ERR_INVALID_ARG for items < 0,
 * k_blocks < 1, units < 1, tiles_per_item not 1 or 2, or NULL outputs.
 */
tgemm_status tgemm_stream_k_plan(int64_t items, int64_t k_blocks, int units, int tiles_per_item,
                                 int64_t *dp_items, int64_t *sk_items, int64_t *sk_units);

/*
 * Diagnostic: the tile order of the persistent scheduler as the GPU computes
 * it.  For every tile number bid of the ceil(M/bm) x ceil(N/bn) grid, one
 * launch writes the tile row to rows[bid] and the tile column to cols[bid],
 * using the device copy of the mapping the GEMM kernels run (the
 * swizzle_2d_from_bid order of "Writing high-performance matrix
 * multiplication with NVIDIA CUDA Tile", section "Performance optimisation:
 * Swizzle"), so that tests can check it against tgemm_tile_coord.
 *   rows, cols  caller-owned device arrays of at least ceil(M/bm) * ceil(N/bn)
 *               int32 elements
 * Asynchronous on `stream`.  Returns TGEMM_ERR_INVALID_ARG for non-positive
 * sizes or NULL arrays, TGEMM_ERR_UNSUPPORTED when tiles * group_m reaches
 * 2^31 (beyond the 32-bit form the kernels use).
 */
tgemm_status tgemm_debug_tile_order(int64_t M, int64_t N, int bm, int bn, int group_m, int32_t *rows, int32_t *cols,
                                    void *stream);

/*
 * Diagnostic: launch one block that waits on a pipeline barrier nobody
 * signals, with a wait limit of `timeout_us` microseconds.  The kernel gives
 * up, records TGEMM_ERR_TIMEOUT's fault code in the status word and returns;
 * tgemm_check(stream) must then report TGEMM_ERR_TIMEOUT and the context
 * stays usable.  This exercises the same bounded-wait routine the GEMM
 * kernels use (the pipeline's "silent deadlock" risk named by the Croqtile
 * tutorial's summary).
 */
tgemm_status tgemm_debug_wait_timeout(uint32_t timeout_us, void *stream);

/*
 * Diagnostic: the same bounded-wait self test (one block, one barrier nobody
 * signals, `timeout_us` microseconds), recording into the status word kept in
 * tgemm_run_noalloc's built-in array instead of the library's own.  It
 * allocates nothing; tgemm_check(stream) must then report TGEMM_ERR_TIMEOUT.
 * Like tgemm_run_noalloc, its first call on a device looks up the array's
 * address, so make it outside CUDA stream capture.  Returns
 * TGEMM_ERR_INVALID_ARG for timeout_us = 0 or above 10 s.
 */
tgemm_status tgemm_debug_noalloc_wait_timeout(uint32_t timeout_us, void *stream);

/*
 * Diagnostic: the SM clock at the moment of the call's turn on `stream`.  One
 * thread counts %clock64 cycles over `duration_us` microseconds of
 * %globaltimer (1 .. 100000) and writes out[0] = the nanoseconds elapsed,
 * out[1] = the cycles counted, so out[1] * 1000 / out[0] is the SM clock in
 * MHz.  out is a caller-owned device array of two uint64_t, 8-byte aligned.
 * Benchmarks place it just before and after a timed region: NVML's clock
 * readings trail the hardware by tens of milliseconds.  The pages report
 * throughput only; this exists so that a throughput can be set against the
 * clock it ran at (per-clock tensor efficiency).
 */
tgemm_status tgemm_debug_sm_clock(uint64_t *out, uint32_t duration_us, void *stream);

/*
 * Diagnostic: record the SM clock inside the GEMM kernels of later calls on
 * the current device.  With `rec` set (a caller-owned device array of eight
 * uint64_t, 8-byte aligned, rec[0..2] zeroed by the caller), every GEMM
 * kernel launched afterwards adds, from its first CTA, the nanoseconds of
 * %globaltimer and the cycles of %clock64 between its dependency wait and its
 * exit to rec[0] and rec[1], and 1 to rec[2] (rec[4..5] are its scratch), so
 * rec[1] * 1000 / rec[0] is the mean SM clock in MHz over those launches.
 * rec = NULL turns it off.  The cost is two stores and three atomics per
 * launch.  Launches captured in a CUDA graph keep the setting they were
 * captured with.  The pages report throughput only; this lets a benchmark set
 * a throughput against the clock it actually ran at: a dense GEMM burst can
 * run well below the clock read just before and just after it.
 */
tgemm_status tgemm_debug_clock_record(uint64_t *rec);

/*
 * tgemm_run without any device allocation, for a skinny A (1..64 rows).
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that may not allocate device memory at call time -- code whose device
 * memory is owned by a pool or budgeted allocator that must see every byte,
 * or that runs where a cudaMalloc would be an error.  tgemm_run allocates a
 * split-K workspace and a status word on first use; this entry point uses a
 * fixed 4 MiB array built into the library instead (reserved on every GPU
 * that loads the library, until the process exits) and never calls
 * cudaMalloc, cudaFree or any allocating routine.
 *
 * Same arguments and result as tgemm_run (C = A * B, same layouts and
 * alignment rules), computed by the same swap-AB split-K kernel, with these
 * limits:
 *   - in_dtype TGEMM_F16 or TGEMM_BF16 (FP8 and FP32 operands return
 *     TGEMM_ERR_UNSUPPORTED);
 *   - 0 <= M <= 64 and N <= 524288 (4096 column tiles of 128); larger sizes
 *     return TGEMM_ERR_UNSUPPORTED before anything is launched;
 *   - every call shares the one array, so calls whose work overlaps on the
 *     GPU (e.g. on two streams without ordering) race and corrupt each
 *     other's results: order them;
 *   - the first call on each device looks up the array's device address
 *     (once); make that first call outside CUDA stream capture;
 *   - a pipeline-wait timeout stops the kernel early and is recorded in a
 *     status word kept in the same array: tgemm_check(stream) then returns
 *     TGEMM_ERR_TIMEOUT (and clears it), as for the other entry points.
 */
tgemm_status tgemm_run_noalloc(int64_t M, int64_t N, int64_t K,
                               const void *A, int64_t lda,
                               const void *B, int64_t ldb, tgemm_b_layout b_layout,
                               void *C, int64_t ldc,
                               tgemm_dtype in_dtype, tgemm_dtype out_dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
