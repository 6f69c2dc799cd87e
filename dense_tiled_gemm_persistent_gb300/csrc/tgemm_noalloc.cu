// tgemm_run_noalloc: the skinny (at most 64 rows of A) swap-AB split-K GEMM
// without any device allocation.
//
// Some callers cannot allocate device memory at the moment they multiply: a
// custom allocator or memory pool owns every byte and forbids cudaMalloc
// behind its back, or the caller runs inside an engine that budgets all
// device memory up front.  tgemm_run allocates its split-K workspace (and a
// status word) with cudaMalloc on first use; this entry point instead keeps
// its workspace in a fixed array that is part of the loaded library image.
//
// The array (kScratchBytes, 4 MiB) is reserved on every GPU that loads the
// library and stays reserved until the process exits.  Layout:
//   [0, 4)                          status word (0 = no fault; zero at load)
//   [4, 256)                        unused
//   [256, 256 + 16 KiB)             per-tile arrival counters (must start at 0)
//   [256 + 16 KiB, kScratchBytes)   FP32 partial sums of the K splits
// Every call uses the same array, so calls whose kernels overlap on the GPU
// (for example on two streams) race on it and give wrong results; callers
// must order them.  Each call clears the counters on its stream before its
// kernel runs; the partial sums need no clearing (every split writes its
// whole slice before anyone reads it).
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in); the device address is looked up once per
// device with cudaGetSymbolAddress, on the first call made while that device
// is current.  That first call should therefore not be made during CUDA
// stream capture.
//
// A kernel that gives up on a pipeline wait winds down as in the other paths
// and records the fault in the array's status word; tgemm_check reads and
// clears it together with the library's own status word.
#include "tgemm.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tgemm_kernel_skinny.cuh"
#include "tgemm_params.h"

#define TGEMM_EXPORT extern "C" __attribute__((visibility("default")))

namespace tgemm {
namespace {

constexpr size_t kScratchBytes = 4u << 20;                 // 4 MiB per GPU
constexpr size_t kReservedBytes = 256;
constexpr size_t kNoAllocCounterBytes = 16u << 10;          // 4096 tiles of 128 columns
constexpr size_t kPartialBytes = kScratchBytes - kReservedBytes - kNoAllocCounterBytes;
constexpr int64_t kMaxRows = 64;                            // M limit of the swap-AB kernel
constexpr int64_t kMaxTiles = (int64_t)(kNoAllocCounterBytes / 4);
constexpr int kMaxDevs = 64;

}  // namespace
}  // namespace tgemm

static __device__ __align__(256) unsigned char g_noalloc_scratch[tgemm::kScratchBytes];

namespace tgemm {
namespace {

std::mutex g_na_mu;
void *g_na_scratch[kMaxDevs];     // device address of g_noalloc_scratch per device
int g_na_sms[kMaxDevs];

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn na_encode_fn()
{
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

bool na_encode(CUtensorMap *map, int dt, const void *ptr, uint64_t inner, uint64_t outer, uint64_t ld,
               uint32_t box_inner, uint32_t box_outer)
{
    EncodeFn enc = na_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t = dt == TGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(map, t, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Set-up for the current device, once: check it is an sm_103 part and look
// up the scratch array's device address.
tgemm_status na_setup(void **scratch, int *sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevs) return TGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (!g_na_scratch[dev]) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        if (!(major == 10 && minor == 3)) return TGEMM_ERR_ARCH;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        g_na_sms[dev] = count;
        g_na_scratch[dev] = p;
    }
    *scratch = g_na_scratch[dev];
    *sms = g_na_sms[dev];
    return TGEMM_OK;
}

const KernelVariant *na_variant(int npad, int out, int w_mn)
{
    const KernelVariant *tab = nullptr;
    int n = 0;
    switch (out) {
    case TGEMM_F16: tab = kVariantsF16; n = kNumVariantsF16; break;
    case TGEMM_BF16: tab = kVariantsBF16; n = kNumVariantsBF16; break;
    case TGEMM_F32: tab = kVariantsF32; n = kNumVariantsF32; break;
    default: return nullptr;
    }
    for (int i = 0; i < n; ++i)
        if (tab[i].cluster == 0 && tab[i].bn == npad && tab[i].b_mn == w_mn) return &tab[i];
    return nullptr;
}

}  // namespace

// The status word of the allocation-free path on device `dev`, or nullptr
// before that path's first call there (tgemm_check reads it).
uint32_t *noalloc_status_word(int dev)
{
    if (dev < 0 || dev >= kMaxDevs) return nullptr;
    std::lock_guard<std::mutex> lk(g_na_mu);
    return static_cast<uint32_t *>(g_na_scratch[dev]);
}

}  // namespace tgemm

using namespace tgemm;

TGEMM_EXPORT tgemm_status tgemm_debug_noalloc_wait_timeout(uint32_t timeout_us, void *stream)
{
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return TGEMM_ERR_INVALID_ARG;
    void *scratch = nullptr;
    int sms = 0;
    tgemm_status st = na_setup(&scratch, &sms);
    if (st != TGEMM_OK) return st;
    if (launch_wait_timeout_probe(static_cast<uint32_t *>(scratch), (uint64_t)timeout_us * 1000ull,
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                                            const void *B, int64_t ldb, tgemm_b_layout b_layout, void *C,
                                            int64_t ldc, tgemm_dtype in_dtype, tgemm_dtype out_dtype,
                                            void *stream)
{
    // ---- host checks, before any CUDA call -------------------------------
    if (b_layout != TGEMM_B_KN && b_layout != TGEMM_B_NK) return TGEMM_ERR_INVALID_ARG;
    if (in_dtype != TGEMM_F16 && in_dtype != TGEMM_BF16) {
        return (in_dtype == TGEMM_F32 || in_dtype == TGEMM_E4M3 || in_dtype == TGEMM_E5M2) ? TGEMM_ERR_UNSUPPORTED
                                                                                           : TGEMM_ERR_INVALID_ARG;
    }
    if (out_dtype != TGEMM_F16 && out_dtype != TGEMM_BF16 && out_dtype != TGEMM_F32) return TGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_ARG;
    // Size limits of this entry point: the swap-AB kernel takes at most 64
    // rows of A, and the counter region holds 4096 column tiles of 128.
    if (M > kMaxRows || ceil_div(N, kSkinnyRows) > kMaxTiles || K >= ((int64_t)1 << 31))
        return TGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return TGEMM_OK;
    const size_t eo = out_dtype == TGEMM_F32 ? 4 : 2;
    if (C == nullptr || ldc < N) return TGEMM_ERR_INVALID_ARG;
    if (((uintptr_t)C % 16) != 0 || ((uint64_t)ldc * eo) % 16 != 0) return TGEMM_ERR_MISALIGNED;
    if (K > 0) {
        if (A == nullptr || B == nullptr || lda < K || ldb < (b_layout == TGEMM_B_KN ? N : K))
            return TGEMM_ERR_INVALID_ARG;
        if (((uintptr_t)A % 16) != 0 || ((uintptr_t)B % 16) != 0 || ((uint64_t)lda * 2) % 16 != 0 ||
            ((uint64_t)ldb * 2) % 16 != 0)
            return TGEMM_ERR_MISALIGNED;
    }

    void *scratch = nullptr;
    int sms = 0;
    tgemm_status st = na_setup(&scratch, &sms);
    if (st != TGEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) {   // the empty sum
        if (cudaMemset2DAsync(C, (size_t)ldc * eo, 0, (size_t)N * eo, (size_t)M, s) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        return TGEMM_OK;
    }

    const int npad = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    const bool w_mn = b_layout == TGEMM_B_KN;
    const KernelVariant *var = na_variant(npad, out_dtype, w_mn ? 1 : 0);
    if (!var) return TGEMM_ERR_UNSUPPORTED;
    const int64_t tiles_n = ceil_div(N, kSkinnyRows);
    const int64_t num_kb = ceil_div(K, kBK);
    // About two CTAs per SM, at most what the partial-sum region holds.
    int64_t splits = (2 * (int64_t)sms + tiles_n / 2) / tiles_n;
    const int64_t per_split = tiles_n * kSkinnyRows * npad * (int64_t)sizeof(float);
    const int64_t fit = (int64_t)kPartialBytes / per_split;
    if (splits > fit) splits = fit;
    if (splits > num_kb) splits = num_kb;
    if (splits > 32) splits = 32;
    if (splits < 1) splits = 1;

    GemmParams p;
    std::memset(&p, 0, sizeof p);
    bool ok = na_encode(&p.tma_a, in_dtype, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, kBK, (uint32_t)npad);
    if (w_mn)
        ok = ok && na_encode(&p.tma_b, in_dtype, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, 64, kBK);
    else
        ok = ok && na_encode(&p.tma_b, in_dtype, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, kBK, kSkinnyRows);
    if (!ok) return TGEMM_ERR_CUDA;
    unsigned char *base = static_cast<unsigned char *>(scratch);
    p.M = (int32_t)M;
    p.N = (int32_t)N;
    p.K = (int32_t)K;
    p.tiles_m = 1;
    p.tiles_n = (int32_t)tiles_n;
    p.num_tiles = (int32_t)tiles_n;
    p.num_kb = (int32_t)num_kb;
    p.group_m = 1;
    p.idesc = make_idesc(in_dtype == TGEMM_BF16, false, kSkinnyRows, npad, w_mn);
    p.status = reinterpret_cast<uint32_t *>(base);   // the array's status word
    const char *env = std::getenv("TGEMM_WAIT_TIMEOUT_MS");
    long ms = env ? std::strtol(env, nullptr, 10) : 0;
    p.timeout_ns = (uint64_t)(ms > 0 ? ms : 2000) * 1000000ull;
    p.c_ptr = C;
    p.ldc = ldc;
    p.splits = (int32_t)splits;
    p.counters = reinterpret_cast<uint32_t *>(base + kReservedBytes);
    p.partials = reinterpret_cast<float *>(base + kReservedBytes + kNoAllocCounterBytes);
    if (splits > 1 &&
        cudaMemsetAsync(p.counters, 0, (size_t)tiles_n * sizeof(uint32_t), s) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    if (var->launch(p, (int)(tiles_n * splits), s) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}
