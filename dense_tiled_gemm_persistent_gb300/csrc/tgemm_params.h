// Kernel parameter block and launch declarations shared by the host API and
// the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace tgemm {

enum OutType { OUT_F16 = 0, OUT_BF16 = 1, OUT_F32 = 2 };

// Fault codes written to the device status word: bits 31..28 hold the
// status (7 = timeout), bits 27..20 the wait site, bits 19..0 the CTA.
enum WaitSite : uint32_t {
    SITE_PRODUCER_EMPTY = 1,
    SITE_MMA_TMEM_EMPTY = 2,
    SITE_MMA_FULL = 3,
    SITE_EPI_TMEM_FULL = 4,
    SITE_DRAIN_LOADS = 5,
    SITE_DRAIN_MMA = 6,
    SITE_DEBUG = 7,
    SITE_SPLITK_COUNTER = 8,
    SITE_EPI_CIN = 9,
    SITE_CLUSTER_EXCHANGE = 10,
};

constexpr uint32_t kFaultTimeout = 7u;

// Everything one persistent GEMM launch needs.  The three tensor maps must
// stay 128-byte aligned (CUtensorMap) inside the parameter space.
// The tile kernels (one CTA, CTA pair) address every operand with 3-D tensor
// maps whose outermost coordinate is the batch (extent 1 when not batched, or
// when the operand is shared by all batches); the skinny kernels use 2-D maps.
struct alignas(128) GemmParams {
    CUtensorMap tma_a;      // A: dims {K, M, batch}, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tma_b;      // B: NK dims {K, N, batch} box {64, bn, 1}; KN dims {N, K, batch} box {64, 64, 1}
    CUtensorMap tma_c;      // C: dims {N, M, batch}, box {128 bytes of columns, 32, 1}, 128-byte swizzle
    CUtensorMap tma_ws;     // stream-K partial tiles (FP32): dims {256, slots * 256, 1}, box {32, 32, 1}
    CUtensorMap tma_cin;    // fused epilogue C_in (output type): same geometry as tma_c
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_tiles, num_kb;
    int32_t tiles_per_batch;   // tiles_m * tiles_n; tile t is batch t / tiles_per_batch
    int32_t a_batched, b_batched;   // 0: the operand is shared by every batch (z = 0)
    int32_t group_m;
    uint32_t idesc;         // tcgen05 instruction descriptor (kind::f16)
    uint32_t *status;       // device status word (first fault wins)
    uint64_t *clock_rec;    // SM-clock record (tgemm_debug_clock_record), or null
    uint64_t timeout_ns;    // limit of every pipeline wait
    // swap-AB / split-K path only
    void *c_ptr;            // C, row-major M x ldc (written with plain stores)
    int64_t ldc;
    float *partials;        // [splits][tiles_n][128 rows][npad] FP32 partial sums
    uint32_t *counters;     // [tiles_n] arrival counters, zero between calls
    int32_t splits;         // K is cut into `splits` runs of whole k-blocks
    int32_t k_alternate;    // pair/quad kernels: odd waves of whole tiles run their K loop backwards
    int32_t prefetch_kb;    // k-blocks of its weight slice a CTA prefetches into L2 before the dependency wait
    int32_t late_trigger;   // 1: let the next launch start once this CTA has issued its last load (else at once)
    // stream-K tail of the CTA-pair kernel (sk_units = 0: whole tiles only)
    int32_t dp_tiles;       // tiles [0, dp_tiles) are processed whole
    int32_t sk_tiles;       // tiles [dp_tiles, dp_tiles + sk_tiles) are spread over
    int32_t sk_units;       // the first sk_units pairs, evenly by k-block
    // fused epilogue D = act(alpha * acc + beta * C_in + bias[column]) before
    // the cast; epi = 0 keeps the plain cast
    float alpha, beta;
    const void *bias;       // N entries or null
    int32_t bias_dtype;     // 0 F16, 1 BF16, 2 F32
    int32_t act;            // 0 none, 1 ReLU, 2 GELU (tanh form)
    int32_t epi;            // bit 0: fused epilogue on; bit 1: read C_in (beta != 0)
    const void *cin_ptr;    // C_in for the kernels that store with plain stores
    int64_t ldc_in;
};

using LaunchFn = cudaError_t (*)(const GemmParams &, int grid, cudaStream_t);
using OccupancyFn = int (*)();

// One compiled kernel variant.  cluster = 1: one CTA per 128 x bn tile;
// cluster = 2: a CTA pair per 256 x bn tile, and max_active reports how many
// pairs fit on the device at once.
struct KernelVariant {
    int bn, stages, out, b_mn;
    size_t smem_bytes;
    LaunchFn launch;
    int cluster;
    OccupancyFn max_active;
    int kind = 0;          // operand kind: 0 FP16/BF16 (kind::f16), 1 FP8 (kind::f8f6f4), 2 TF32 (kind::tf32)
};

// Defined in the kernel translation units (one per output type).
extern const KernelVariant kVariantsF16[];
extern const int kNumVariantsF16;
extern const KernelVariant kVariantsBF16[];
extern const int kNumVariantsBF16;
extern const KernelVariant kVariantsF32[];
extern const int kNumVariantsF32;

// Raise a kernel's dynamic shared-memory limit once per device (the
// attribute is per device and costs a driver call; launches are frequent).
template <class Kernel>
inline cudaError_t ensure_smem_limit(Kernel kern, unsigned smem, std::atomic<unsigned long long> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// The bounded-wait self test and SM-clock probe launchers (tgemm_debug.cu).
cudaError_t launch_wait_timeout_probe(uint32_t *status, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_sm_clock_probe(uint64_t *out, uint64_t duration_ns, cudaStream_t st);
// tgemm_noalloc.cu: the allocation-free path's status word on a device
// (nullptr before that path's first call there)
uint32_t *noalloc_status_word(int dev);

}  // namespace tgemm
