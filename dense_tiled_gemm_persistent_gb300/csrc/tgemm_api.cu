// Host side of the C ABI declared in include/tgemm.h: argument validation,
// configuration choice, tensor-map encoding and the launch of the persistent
// kernels.  Nothing here computes any part of C; every element of the result
// is produced by the device kernels (or, for K = 0, by a device memset that
// writes the empty sum).
#include "tgemm.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>

#include "tgemm_kernel_pair.cuh"
#include "tgemm_kernel_skinny.cuh"
#include "tgemm_kernel_splitk_cluster.cuh"
#include "tgemm_params.h"
#include "tgemm_sched.h"

#define TGEMM_EXPORT extern "C" __attribute__((visibility("default")))

namespace tgemm {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultGroupM = 8;   // GROUP_SIZE_M of the cuTile tutorial's matmul example

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *status = nullptr;     // device status word, lazily allocated
    std::map<const void *, int> pairs;   // resident CTA pairs per pair-kernel variant
    std::atomic<uint64_t *> clock_rec{nullptr};   // tgemm_debug_clock_record's buffer, or null
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Split-K workspace, one per (device, stream) so that calls on different
// streams never share partial sums: [counters: kCounterBytes][partials].
constexpr size_t kCounterBytes = 64 * 1024;        // 16384 tile counters
constexpr int kMaxSkinnyTiles = (int)(kCounterBytes / 4);
struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::map<std::pair<int, void *>, Workspace> g_ws;
std::atomic<uint32_t> g_last_fault{0};   // last non-zero status word seen by tgemm_check

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

uint64_t wait_timeout_ns()
{
    static uint64_t ns = [] {
        const char *s = std::getenv("TGEMM_WAIT_TIMEOUT_MS");
        long ms = s ? std::strtol(s, nullptr, 10) : 0;
        if (ms <= 0) ms = 2000;
        return (uint64_t)ms * 1000000ull;
    }();
    return ns;
}

size_t elem_size(int dt) { return dt == TGEMM_F32 ? 4 : (dt == TGEMM_E4M3 || dt == TGEMM_E5M2) ? 1 : 2; }
bool is_f8(int dt) { return dt == TGEMM_E4M3 || dt == TGEMM_E5M2; }
// Operands that only the tile kernels take (K-major B): FP8, and FP32 read as TF32.
bool tile_only(int dt) { return is_f8(dt) || dt == TGEMM_F32; }
int mma_kind(int in_dtype) { return is_f8(in_dtype) ? KIND_F8 : in_dtype == TGEMM_F32 ? KIND_TF32 : KIND_F16; }

// Whether a swap-AB mode (0 none, 1 workspace, 2 in-cluster) has kernels for
// this operand type: both for FP16/BF16, the in-cluster one for FP8, none for
// FP32 read as TF32.
bool swap_supported(int in_dtype, int swap_ab)
{
    if (swap_ab == 0) return true;
    if (is_f8(in_dtype)) return swap_ab == 2;
    return !tile_only(in_dtype);
}
// K elements in one 128-byte k-block row
int kblock_elems(int in_dtype) { return (int)(128 / elem_size(in_dtype)); }
// Instruction-descriptor operand type: kind::f16 0 F16 / 1 BF16, kind::f8f6f4
// 0 E4M3 / 1 E5M2, kind::tf32 2.
uint32_t mma_type(int in_dtype)
{
    return in_dtype == TGEMM_F32 ? 2u : (in_dtype == TGEMM_BF16 || in_dtype == TGEMM_E5M2) ? 1u : 0u;
}

// Current device's state; allocates the status word on first use.
tgemm_status device_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return TGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        d.ready = true;
    }
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return TGEMM_ERR_ARCH;
    if (!d.status) {
        void *p = nullptr;
        if (cudaMalloc(&p, sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_OOM;
        }
        if (cudaMemset(p, 0, sizeof(uint32_t)) != cudaSuccess) {
            cudaFree(p);
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        d.status = static_cast<uint32_t *>(p);
    }
    *out = &d;
    return TGEMM_OK;
}

// Host-only checks (no CUDA call).  Returns TGEMM_OK with *noop set when
// there is nothing to compute (M = 0 or N = 0).
tgemm_status validate(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                      int64_t ldb, int b_layout, const void *C, int64_t ldc, int in_dtype, int out_dtype,
                      bool *noop)
{
    *noop = false;
    if (b_layout != TGEMM_B_KN && b_layout != TGEMM_B_NK) return TGEMM_ERR_INVALID_ARG;
    if (in_dtype != TGEMM_F16 && in_dtype != TGEMM_BF16 && in_dtype != TGEMM_F32 && !is_f8(in_dtype))
        return TGEMM_ERR_INVALID_ARG;
    if (out_dtype != TGEMM_F16 && out_dtype != TGEMM_BF16 && out_dtype != TGEMM_F32)
        return TGEMM_ERR_INVALID_ARG;
    if (tile_only(in_dtype) && b_layout != TGEMM_B_NK) return TGEMM_ERR_UNSUPPORTED;   // FP8/TF32: K-major B only
    if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_ARG;
    // Tensor coordinates are signed 32-bit.
    const int64_t kMax = (int64_t)1 << 31;
    if (M >= kMax || N >= kMax || K >= kMax) return TGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) {
        *noop = true;
        return TGEMM_OK;
    }
    if (ldc < N) return TGEMM_ERR_INVALID_ARG;
    if (C == nullptr) return TGEMM_ERR_INVALID_ARG;
    const size_t ei = elem_size(in_dtype), eo = elem_size(out_dtype);
    if (((uintptr_t)C % 16) != 0 || ((uint64_t)ldc * eo) % 16 != 0) return TGEMM_ERR_MISALIGNED;
    if (K == 0) return TGEMM_OK;
    if (lda < K) return TGEMM_ERR_INVALID_ARG;
    if (ldb < (b_layout == TGEMM_B_KN ? N : K)) return TGEMM_ERR_INVALID_ARG;
    if (A == nullptr || B == nullptr) return TGEMM_ERR_INVALID_ARG;
    if (((uintptr_t)A % 16) != 0 || ((uintptr_t)B % 16) != 0) return TGEMM_ERR_MISALIGNED;
    if (((uint64_t)lda * ei) % 16 != 0 || ((uint64_t)ldb * ei) % 16 != 0) return TGEMM_ERR_MISALIGNED;
    return TGEMM_OK;
}

const KernelVariant *find_variant(int bn, int stages, int out, int b_mn, int cluster, int kind = KIND_F16)
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
        if (tab[i].bn == bn && tab[i].stages == stages && tab[i].b_mn == b_mn && tab[i].cluster == cluster &&
            tab[i].kind == kind)
            return &tab[i];
    return nullptr;
}

// CTAs of a one-CTA tile variant resident per SM (the kernels' TileResidency).
int tile_ctas_per_sm(int bn, int stages)
{
    return (bn == 128 && stages <= 2) ? TileResidency<128, 2>::ctas_per_sm : 1;
}

void fill_config(tgemm_config *cfg, int cluster, int bn, int64_t tiles, int units)
{
    cfg->bm = cluster == 2 ? kPairBM : kBM;
    cfg->bn = bn;
    cfg->bk = kBK;
    cfg->stages = cluster == 2 ? 6 : (bn == 256 ? 4 : 6);
    cfg->cluster_m = cluster;
    cfg->group_m = kDefaultGroupM;
    cfg->split_k = 1;
    cfg->swap_ab = 0;
    const int64_t ctas = (tiles < units ? tiles : units) * cluster;
    cfg->grid = (int)ctas;
}

// Rows of A a swap-AB kernel pads to (its MMA's N); 128 only in the
// in-cluster kernel (65 to 128 rows).
int skinny_npad(int64_t M) { return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128)); }
constexpr int64_t kMaxSwapRows = 128;

// Splits of the K loop for the swap-AB path: about two CTAs per SM stream
// the weights, every split keeps at least one k-block.
int skinny_splits(int64_t N, int64_t K, int sm_count)
{
    const int64_t tiles = ceil_div(N, kSkinnyRows);
    const int64_t kb = ceil_div(K, kBK);
    if (tiles > kMaxSkinnyTiles) return 1;
    int64_t s = (2 * sm_count + tiles / 2) / tiles;
    if (s > kb) s = kb;
    if (s > 32) s = 32;
    if (s < 1) s = 1;
    return (int)s;
}

// Tile-shape choice by a wave cost model: time ~ waves * (per-SM time of one
// tile).  A CTA of the pair kernel and a 128 x 256 one-CTA tile do the same
// MMA work per SM, but the pair moves a third fewer operand bytes per SM;
// a 128 x 128 tile halves the work per SM for 2/3 of the bytes of a
// 128 x 256 one and keeps the tensor pipe less busy.  At most 64 rows of A
// go to the swap-AB split-K path instead.
// Measured winners per grid point (tune_picker.py); the last row is a sentinel.
// Operand classes have rows of their own: 0 = FP16/BF16, 1 = FP8, 2 = FP32
// read as TF32 (the last two measured with B stored N x K, the only layout
// their kernels take, and more than 64 rows of A).
struct PickRow {
    int em, en, ek, layout, dclass;
    struct { int bm, bn, stages, cluster_m, group_m, split_k, swap_ab; } c;
    float us;
};
const PickRow kPickTable[] = {
#include "tgemm_picker_table.inc"
    {-1, -1, -1, -1, -1, {0, 0, 0, 0, 0, 0, 0}, 0.f},
};

int pick_class(int in_dtype) { return is_f8(in_dtype) ? 1 : in_dtype == TGEMM_F32 ? 2 : 0; }

int round_log2(int64_t x)
{
    int e = 0;
    while (((int64_t)1 << (e + 1)) <= x) ++e;            // floor(log2 x)
    // round: x >= 2^(e + 0.5)  <=>  x^2 >= 2^(2e + 1)
    const double xd = (double)x;
    return (xd * xd >= (double)((int64_t)1 << (2 * e + 1))) ? e + 1 : e;
}

// The measured winner at the grid point nearest (in log2) to this shape, if
// the table has one; its tile shape and split are kept, sizes re-derived.
// Grid point -> table row, built once: a linear scan of the ~1500 rows cost
// microseconds of host time per call.
int table_row(int em, int en, int ek, int layout, int dclass)
{
    auto key = [](int em_, int en_, int ek_, int layout_, int dclass_) {
        return ((((uint64_t)(uint32_t)dclass_ * 2 + (uint32_t)layout_) * 64 + (uint32_t)em_) * 64 + (uint32_t)en_) *
                   64 + (uint32_t)ek_;
    };
    static const std::map<uint64_t, int> index = [&] {
        std::map<uint64_t, int> m;
        for (int i = 0; kPickTable[i].em >= 0; ++i) {
            const PickRow &r = kPickTable[i];
            m.emplace(key(r.em, r.en, r.ek, r.layout, r.dclass), i);
        }
        return m;
    }();
    if (em < 0 || em >= 64 || en < 0 || en >= 64 || ek < 0 || ek >= 64) return -1;
    const auto it = index.find(key(em, en, ek, layout, dclass));
    return it == index.end() ? -1 : it->second;
}

bool table_config(int64_t M, int64_t N, int64_t K, int b_layout, int dclass, int sm_count, tgemm_config *cfg)
{
    const int row = table_row(round_log2(M), round_log2(N), round_log2(K), b_layout, dclass);
    if (row >= 0) {
        const PickRow &r = kPickTable[row];
        cfg->bm = r.c.bm;
        cfg->bn = r.c.bn;
        cfg->bk = kBK;
        cfg->stages = r.c.stages;
        cfg->cluster_m = r.c.cluster_m;
        cfg->group_m = r.c.group_m;
        cfg->split_k = r.c.split_k;
        cfg->swap_ab = r.c.swap_ab;
        cfg->grid = 0;
        if (cfg->swap_ab) {
            if (M > kMaxSwapRows) return false;
            if (skinny_npad(M) != cfg->bn) return false;   // grid point of another padding class
        } else if (M <= 64) {
            return false;
        }
        (void)sm_count;
        return true;
    }
    return false;
}

// Largest split count of the in-cluster kernel: an owner's ring receives
// the other ranks' partials of its quarters, bounded by S-1 whole partials
// (the half-size ring, named by its stage count, holds fewer).
template <int NPAD>
int cluster_splits_limit_of(int stages)
{
    return stages == ClusterSplitPlan<NPAD, 108>::stages ? ClusterSplitPlan<NPAD, 108>::max_splits
                                                         : ClusterSplitPlan<NPAD>::max_splits;
}
int cluster_splits_limit(int npad, int stages = 0)
{
    return npad == 16 ? cluster_splits_limit_of<16>(stages)
           : npad == 32 ? cluster_splits_limit_of<32>(stages)
           : npad == 64 ? cluster_splits_limit_of<64>(stages) : ClusterSplitPlan<128>::max_splits;
}
int cluster_stages(int npad)
{
    return npad == 16 ? ClusterSplitPlan<16>::stages
           : npad == 32 ? ClusterSplitPlan<32>::stages
           : npad == 64 ? ClusterSplitPlan<64>::stages : ClusterSplitPlan<128>::stages;
}

void choose_config_model(int64_t M, int64_t N, int64_t K, int sm_count, tgemm_config *cfg, int64_t batch = 1,
                         bool allow_swap = true, int dclass = 0);

// CTAs of a quad launch (four per quad): one quad per 256 x 512 block with
// whole blocks, every quad with a stream-K tail; resident limits apply later.
int quad_grid(int64_t M, int64_t N, int split_k, int sm_count)
{
    const int64_t blocks = ceil_div(M, kPairBM) * ceil_div(ceil_div(N, kPairBN), 2);
    const int64_t quads = split_k == 0 ? sm_count / 4 : std::min<int64_t>(blocks, sm_count / 4);
    return (int)(4 * std::max<int64_t>(quads, 1));
}

// The configuration tgemm_run uses: the measured table where it covers the
// shape and its entry is legal for it, the wave cost model otherwise.
void choose_config(int64_t M, int64_t N, int64_t K, int b_layout, int dclass, int sm_count, tgemm_config *cfg)
{
    if (table_config(M, N, K, b_layout, dclass, sm_count, cfg)) {
        const int64_t kb = ceil_div(K, kBK);
        bool ok = cfg->split_k <= kb;
        if (ok && cfg->swap_ab == 2) ok = cfg->split_k <= cluster_splits_limit(cfg->bn, cfg->stages);
        if (ok) {
            if (cfg->swap_ab)
                cfg->grid = (int)(ceil_div(N, kSkinnyRows) * cfg->split_k);
            else if (cfg->cluster_m == 2)
                cfg->grid = cfg->split_k == 0 ? 2 * (sm_count / 2)
                                              : (int)(2 * std::min<int64_t>(TileGrid(M, N, cfg->bm, cfg->bn).count(),
                                                                            sm_count / 2));
            else if (cfg->cluster_m == 4)
                cfg->grid = quad_grid(M, N, cfg->split_k, sm_count);
            else
                cfg->grid = (int)std::min<int64_t>(TileGrid(M, N, cfg->bm, cfg->bn).count(),
                                                   (int64_t)sm_count * tile_ctas_per_sm(cfg->bn, cfg->stages));
            return;
        }
    }
    choose_config_model(M, N, K, sm_count, cfg, 1, true, dclass);
}

void choose_config_model(int64_t M, int64_t N, int64_t K, int sm_count, tgemm_config *cfg, int64_t batch,
                         bool allow_swap, int dclass)
{
    // Operand classes: 0 FP16/BF16 (every kernel), 1 FP8 (the tile kernels
    // and the in-cluster swap-AB kernel), 2 TF32 (the tile kernels).
    if (dclass == 2) allow_swap = false;
    const bool two_stage = dclass == 0;
    const int64_t kbe = dclass == 1 ? KBlock<KIND_F8>::elems : kBK;   // K elements per 128-byte k-block
    if (allow_swap && M > 64 && M <= kMaxSwapRows && 2 * ceil_div(N, kSkinnyRows) <= sm_count) {
        // 65-128 rows: the in-cluster kernel padded to 128 (one 128 x 128 x
        // 16 MMA per 16 of K) where the weight's column tiles leave room for
        // at least two splits each; the ring holds three 64 KiB partials, so
        // at most four splits.  Measured on one GB300 (BF16, graph-replayed):
        // 128 x 4096 x 4096 20.1 -> 14.6 us against 128 x 128 tiles,
        // 128 x 4096 x 14336 51.4 -> 30.4 us against pair + stream-K, 128 x
        // 1024 x 4096 19.7 -> 12.1 us; with one split (128 x 14336 x 4096,
        // 112 column tiles) it was 11 % slower than the tiles.
        const int64_t tiles = ceil_div(N, kSkinnyRows);
        const int64_t kb = ceil_div(K, kbe);
        int64_t cs = sm_count / tiles;
        if (cs > ClusterSplitPlan<128>::max_splits) cs = ClusterSplitPlan<128>::max_splits;
        if (cs > kb) cs = kb;
        if (cs < 1) cs = 1;
        cfg->bm = kSkinnyRows;
        cfg->bn = 128;
        cfg->bk = kBK;
        cfg->stages = ClusterSplitPlan<128>::stages;
        cfg->cluster_m = (int)cs;
        cfg->group_m = 1;
        cfg->split_k = (int)cs;
        cfg->swap_ab = 2;
        cfg->grid = (int)(tiles * cs);
        return;
    }
    if (allow_swap && M <= 64) {
        const int npad = skinny_npad(M);
        const int64_t tiles = ceil_div(N, kSkinnyRows);
        const int64_t kb = ceil_div(K, kbe);
        // In-cluster split-K: one CTA per SM, the splits of a tile reduce
        // through distributed shared memory.  Used unless the tiles are so few
        // that the cluster limit leaves most SMs idle.  For up to 16 rows the
        // half-size ring (two CTAs per SM) measured faster across the tuning
        // grid; its second slot per SM lets up to sm_count tiles split in two.
        const bool half = npad == 16;
        const int stages = half ? ClusterSplitPlan<16, 108>::stages : cluster_stages(npad);
        const int limit = cluster_splits_limit(npad, stages);
        int64_t cs = sm_count / (tiles > 0 ? tiles : 1);
        if (half && cs < 2 && tiles <= sm_count) cs = 2;
        if (cs > limit) cs = limit;
        if (cs > kb) cs = kb;
        if (cs < 1) cs = 1;
        cfg->bm = kSkinnyRows;
        cfg->bn = npad;
        cfg->bk = kBK;
        cfg->group_m = 1;
        if (2 * tiles * cs >= sm_count || cs == kb || dclass == 1) {   // (no FP8 workspace kernel)
            cfg->stages = stages;
            cfg->cluster_m = (int)cs;
            cfg->split_k = (int)cs;
            cfg->swap_ab = 2;
            cfg->grid = (int)(tiles * cs);
            return;
        }
        const int s = skinny_splits(N, K, sm_count);
        cfg->stages = kSkinnyStages;
        cfg->cluster_m = 1;
        cfg->split_k = s;
        cfg->swap_ab = 1;
        cfg->grid = (int)(tiles * s);
        return;
    }
    // Time of one tile on its SM(s), in cycles: the mainloop (8 cycles per
    // element of K for a 128 x 256 half-tile at full MMA rate, the pair's
    // at 0.85 of that per SM, 128 x 128 tiles at 1.25x per column) or a
    // floor for draining the accumulator and storing the tile (3000 cycles
    // for 128 x 256, half for 128 x 128), whichever is longer: the two
    // overlap through the double TMEM accumulator.  Short K (many small
    // batched problems) hits the floor, where finer tiles fill the waves
    // better.  The floor puts the crossover where batches of 512 x 512
    // products measured it on a GB300: 128 x 128 tiles ahead at K = 128
    // (12.5 against 14.0 us for 64 of them), CTA pairs ahead at K = 512
    // (20.9 against 23.7 us).
    //
    // With one k-block per tile (K <= 64) the two-stage 128 x 128 ring, two
    // CTAs per SM (each at half the SM's MMA rate), doubles the tiles in
    // flight and the epilogue warps: measured on one GB300, 64 x 512x512x64
    // 11.5 -> 9.6 us and 128 x 256x256x64 8.5 -> 7.3 us against the six-stage
    // ring; at K = 128 the two were within 2 %, beyond it the six stages won
    // (64 x 512x512x256 15.2 against 20.3 us).  16-bit operands only.
    struct Cand { int cluster, bn; double main_per_k, epi; int stages, per_sm; };
    // (on a tie the one-CTA tiles: more CTAs in flight for the same waves)
    const Cand cands[] = {{1, 256, 8, 3000, 4, 1}, {1, 128, 1.25 * 4, 1500, 6, 1}, {2, 256, 0.85 * 8, 3000, 6, 1},
                          {1, 128, 2 * 1.25 * 4, 1500, 2, 2}};
    const int n_cands = (two_stage && K <= kBK) ? 4 : 3;
    double best = 0;
    const Cand *pick = nullptr;
    int64_t pick_tiles = 0;
    int pick_units = 0;
    for (int ci = 0; ci < n_cands; ++ci) {
        const Cand &c = cands[ci];
        const int bm = c.cluster == 2 ? kPairBM : kBM;
        const TileGrid g(M, N, bm, c.bn);
        const int units = (c.cluster == 2 ? sm_count / 2 : sm_count) * c.per_sm;
        const double per_tile = std::max(c.main_per_k * (double)K, c.epi);
        const double cost = (double)ceil_div(g.count() * batch, units) * per_tile;
        if (!pick || cost < best) {
            pick = &c;
            best = cost;
            pick_tiles = g.count();
            pick_units = units;
        }
    }
    fill_config(cfg, pick->cluster, pick->bn, pick_tiles, pick_units);
    cfg->stages = pick->stages;
    // Few pair tiles over a deep K leave most pairs idle: share the K loop
    // out (stream-K) when at most half the pairs would get a tile.
    if (pick->cluster == 2 && 2 * pick_tiles <= pick_units && ceil_div(K, kBK) >= 64) {
        cfg->split_k = 0;
        cfg->grid = 2 * pick_units;
    }
}

CUtensorMapDataType map_dtype(int dt)
{
    switch (dt) {
    case TGEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case TGEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case TGEMM_E4M3:
    case TGEMM_E5M2: return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // the copy engine only moves bytes
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    }
}

// 2-D row-major tensor: `inner` contiguous elements per row, `outer` rows,
// `ld` elements between rows; boxes of box_inner x box_outer, 128-byte swizzle,
// zero fill outside the tensor.
// Row-major tensor of `outer` rows of `inner` elements, `ld` elements apart;
// rank 3 adds `batch` copies `bstride` elements apart (the outermost
// coordinate).  Boxes of box_inner x box_outer (x 1), 128-byte swizzle, zero
// fill outside the tensor.
bool encode_map_uncached(CUtensorMap *map, int dt, const void *ptr, int rank, uint64_t inner, uint64_t outer,
                         uint64_t ld, uint64_t batch, uint64_t bstride, uint32_t box_inner, uint32_t box_outer)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const size_t e = elem_size(dt);
    const cuuint64_t dims[3] = {inner, outer, batch};
    const cuuint64_t strides[2] = {ld * e, bstride * e};
    const cuuint32_t box[3] = {box_inner, box_outer, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, map_dtype(dt), (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A small direct-mapped cache of encoded tensor maps: a descriptor depends
// only on (address, type, rank, extents, pitches, box), so repeated calls on
// the same buffers skip the driver's encoder.
struct MapKey {
    const void *ptr;
    int dt, rank;
    uint64_t inner, outer, ld, batch, bstride;
    uint32_t box_inner, box_outer;
    bool operator==(const MapKey &o) const
    {
        return ptr == o.ptr && dt == o.dt && rank == o.rank && inner == o.inner && outer == o.outer && ld == o.ld &&
               batch == o.batch && bstride == o.bstride && box_inner == o.box_inner && box_outer == o.box_outer;
    }
};
struct MapSlot {
    bool valid = false;
    MapKey key;
    CUtensorMap map;
};
constexpr int kMapSlots = 256;
std::mutex g_map_mu;
MapSlot g_maps[kMapSlots];

bool encode_map(CUtensorMap *map, int dt, const void *ptr, int rank, uint64_t inner, uint64_t outer, uint64_t ld,
                uint64_t batch, uint64_t bstride, uint32_t box_inner, uint32_t box_outer)
{
    if (rank == 2) {
        batch = 1;
        bstride = 0;
    }
    const MapKey key{ptr, dt, rank, inner, outer, ld, batch, bstride, box_inner, box_outer};
    uint64_t h = (uint64_t)(uintptr_t)ptr * 0x9E3779B97F4A7C15ull;
    h ^= (inner * 31 + outer + (uint64_t)rank * 7) * 0xC2B2AE3D27D4EB4Full;
    h ^= (ld + ((uint64_t)box_inner << 20) + ((uint64_t)box_outer << 40) + (uint64_t)dt) * 0x165667B19E3779F9ull;
    h ^= (batch * 131 + bstride) * 0x27D4EB2F165667C5ull;
    MapSlot &slot = g_maps[(h >> 32) % kMapSlots];
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        if (slot.valid && slot.key == key) {
            *map = slot.map;
            return true;
        }
    }
    if (!encode_map_uncached(map, dt, ptr, rank, inner, outer, ld, batch, bstride, box_inner, box_outer)) return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    slot.valid = true;
    slot.key = key;
    slot.map = *map;
    return true;
}

bool encode_2d(CUtensorMap *map, int dt, const void *ptr, uint64_t inner, uint64_t outer, uint64_t ld,
               uint32_t box_inner, uint32_t box_outer)
{
    return encode_map(map, dt, ptr, 2, inner, outer, ld, 1, 0, box_inner, box_outer);
}

// The 3-D map of one operand of the tile kernels: `batch` copies `bstride`
// elements apart, or one copy shared by every batch (bstride = 0).
bool encode_3d(CUtensorMap *map, int dt, const void *ptr, uint64_t inner, uint64_t outer, uint64_t ld,
               uint64_t batch, uint64_t bstride, uint32_t box_inner, uint32_t box_outer)
{
    if (bstride == 0) {
        batch = 1;
        bstride = ld * outer;   // any legal pitch: the single copy is never stepped over
    }
    return encode_map(map, dt, ptr, 3, inner, outer, ld, batch, bstride, box_inner, box_outer);
}

// Batch description of a call (count 1: not batched).  Strides in elements.
struct Batch {
    int64_t count = 1, sa = 0, sb = 0, sc = 0;
};

tgemm_status legal_config(const tgemm_config &c, int64_t M, int64_t K, int out_dtype, int b_layout,
                          const KernelVariant **v, int in_dtype = TGEMM_F16)
{
    if (c.bk != kBK || c.grid < 0 || c.group_m < 1) return TGEMM_ERR_UNSUPPORTED;
    if (tile_only(in_dtype)) {
        // FP8 / TF32: the tile kernels, K-major B (bk names the 128-byte k-block)
        if (b_layout != TGEMM_B_NK) return TGEMM_ERR_UNSUPPORTED;
        if (c.swap_ab == 2 && is_f8(in_dtype)) {
            // FP8 in-cluster swap-AB split-K (128 K elements per k-block)
            const int64_t kb = ceil_div(K > 0 ? K : 1, (int64_t)KBlock<KIND_F8>::elems);
            if (c.bm != kSkinnyRows || c.bn < M || c.cluster_m != c.split_k || c.split_k < 1 || c.split_k > kb)
                return TGEMM_ERR_UNSUPPORTED;
            *v = find_variant(c.bn, c.stages, out_dtype, 0, 3, KIND_F8);
            if (!*v || c.split_k > (*v)->max_active()) return TGEMM_ERR_UNSUPPORTED;
            return TGEMM_OK;
        }
        if (c.swap_ab != 0) return TGEMM_ERR_UNSUPPORTED;
        if (!(c.split_k == 1 || (c.split_k == 0 && (c.cluster_m == 2 || c.cluster_m == 4))))
            return TGEMM_ERR_UNSUPPORTED;
        if (!((c.cluster_m == 1 && c.bm == kBM) ||
              ((c.cluster_m == 2 || c.cluster_m == 4) && c.bm == kPairBM && c.bn == kPairBN)))
            return TGEMM_ERR_UNSUPPORTED;
        *v = find_variant(c.bn, c.stages, out_dtype, 0, c.cluster_m, mma_kind(in_dtype));
        return *v ? TGEMM_OK : TGEMM_ERR_UNSUPPORTED;
    }
    const int b_mn = b_layout == TGEMM_B_KN ? 1 : 0;
    if (c.swap_ab == 1) {
        // swap-AB, split-K through a global workspace: bm weight rows per
        // CTA, bn = padded row count of A (>= M)
        if (c.bm != kSkinnyRows || c.cluster_m != 1 || c.stages != kSkinnyStages) return TGEMM_ERR_UNSUPPORTED;
        if (c.bn < M || c.split_k < 1 || c.split_k > 1024 || c.split_k > ceil_div(K > 0 ? K : 1, kBK))
            return TGEMM_ERR_UNSUPPORTED;
        *v = find_variant(c.bn, c.stages, out_dtype, b_mn, 0);
        return *v ? TGEMM_OK : TGEMM_ERR_UNSUPPORTED;
    }
    if (c.swap_ab == 2) {
        // swap-AB, split-K inside a cluster of split_k CTAs
        if (c.bm != kSkinnyRows || c.bn < M || c.cluster_m != c.split_k || c.split_k < 1 ||
            c.split_k > ceil_div(K > 0 ? K : 1, kBK))
            return TGEMM_ERR_UNSUPPORTED;
        *v = find_variant(c.bn, c.stages, out_dtype, b_mn, 3);
        if (!*v || c.split_k > (*v)->max_active()) return TGEMM_ERR_UNSUPPORTED;
        return TGEMM_OK;
    }
    if (c.swap_ab != 0) return TGEMM_ERR_UNSUPPORTED;
    // split_k = 0 asks the pair or quad kernel for a stream-K tail; cluster_m
    // = 4 is two pairs sharing A (256 x 256 per pair)
    if (!(c.split_k == 1 || (c.split_k == 0 && (c.cluster_m == 2 || c.cluster_m == 4))))
        return TGEMM_ERR_UNSUPPORTED;
    if (!((c.cluster_m == 1 && c.bm == kBM) || ((c.cluster_m == 2 || c.cluster_m == 4) && c.bm == kPairBM &&
                                                c.bn == kPairBN)))
        return TGEMM_ERR_UNSUPPORTED;
    *v = find_variant(c.bn, c.stages, out_dtype, b_mn, c.cluster_m);
    return *v ? TGEMM_OK : TGEMM_ERR_UNSUPPORTED;
}

// The split-K workspace of (current device, stream), grown on demand; the
// counter region is zeroed (stream-ordered) whenever it is (re)allocated and
// is kept zero by the kernels themselves.
tgemm_status split_workspace(int dev, void *stream, size_t partial_bytes, uint32_t **counters, float **partials)
{
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_ws[std::make_pair(dev, stream)];
    const size_t need = kCounterBytes + partial_bytes;
    if (w.bytes < need) {
        if (w.ptr) {
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        void *p = nullptr;
        if (cudaMalloc(&p, need) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_OOM;
        }
        if (cudaMemsetAsync(p, 0, kCounterBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
            cudaFree(p);
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        w.ptr = p;
        w.bytes = need;
    }
    *counters = static_cast<uint32_t *>(w.ptr);
    *partials = reinterpret_cast<float *>(static_cast<char *>(w.ptr) + kCounterBytes);
    return TGEMM_OK;
}

// Resident clusters (CTA pairs, or quads) for a cluster-kernel variant on
// this device (cached).
int resident_pairs(DeviceState *dev, const KernelVariant *v)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = dev->pairs.find((const void *)v);
    if (it != dev->pairs.end()) return it->second;
    int n = v->max_active ? v->max_active() : 0;
    if (n <= 0) n = dev->sm_count / 2;
    dev->pairs[(const void *)v] = n;
    return n;
}

// Stream-K tail for the pair and quad kernels: when the work items (pair
// tiles, or the quad's 256 x 512 blocks of tiles_per_item = 2 tiles) leave
// the last wave partly idle, the last one or two waves' items are shared out
// by k-block iterations (at least kMinSkIters per unit, at most kMaxSegments
// items touched per unit).  Fills p.dp_tiles/sk_tiles/sk_units, the FP32
// partial-tile workspace and its tensor map; sk_units = 0 keeps whole items.
// The quad shares only a leftover wave that is at most half full: sharing a
// full wave as well measured 3-5 % slower than whole blocks on 4000 x 3000 x
// 5000 and 4096 x 3072 x 5000 (96 blocks on 36 quads), where the FP32
// partials of 60 shared blocks cost more than the idle third of a wave.
constexpr int64_t kMinSkIters = 8;

// The split itself, without allocation: T items of KB k-blocks over P units.
// Returns false to keep whole items; otherwise dp whole items come first and
// the sk_items after them are shared by `units` units in equal shares of
// k-block iterations.  tgemm_stream_k_plan exposes it to host tests.
bool stream_k_split(int64_t T, int64_t KB, int64_t P, int tiles_per_item, int64_t *dp_out, int64_t *sk_out,
                    int64_t *units_out)
{
    if (T <= 0 || KB <= 0 || P <= 0) return false;
    const int64_t full = T / P, rem = T % P;
    if (rem == 0) return false;
    int64_t dp, sk_tiles, units;
    if (full >= 1 && 2 * rem <= P) {
        // The leftover wave is at most half full: keep every full wave whole
        // and cut each leftover tile into s = P / rem equal k-ranges, one per
        // pair, so the tail takes 1/s of a tile's time.
        dp = full * P;
        sk_tiles = rem;
        units = (P / rem) * rem;
        if (KB / (P / rem) < kMinSkIters) units = (KB / kMinSkIters) * rem;
        if (units > P) units = P;
    } else {
        // Share the last full wave and the leftover tiles among all pairs.
        if (tiles_per_item > 1 && full >= 1) return false;
        dp = full >= 1 ? (full - 1) * P : 0;
        sk_tiles = T - dp;
        units = sk_tiles * KB / kMinSkIters;
        if (units > P) units = P;
    }
    if (units <= sk_tiles && full == 0) return false;   // no more pairs than tiles to share with
    if (units < 2) return false;
    // never a longer critical path than whole items (shallow K: shares held
    // at kMinSkIters iterations can exceed one item's k-blocks)
    if ((dp / P) * KB + ceil_div(sk_tiles * KB, units) > ceil_div(T, P) * KB) return false;
    if (2 * tiles_per_item * sk_tiles * 4 > (int64_t)kCounterBytes) return false;
    const StreamK sk{sk_tiles, units, KB};
    for (int64_t u = 0; u < units; ++u) {
        if (sk.bound(u + 1) <= sk.bound(u)) return false;                 // empty share
        const int64_t segs = (sk.bound(u + 1) - 1) / KB - sk.bound(u) / KB + 1;
        if (segs > kMaxSegments) return false;
    }
    *dp_out = dp;
    *sk_out = sk_tiles;
    *units_out = units;
    return true;
}

tgemm_status plan_stream_k(GemmParams *p, int pairs, DeviceState *dev, void *stream_ptr, int tiles_per_item = 1)
{
    (void)dev;
    p->dp_tiles = p->num_tiles;
    p->sk_tiles = 0;
    p->sk_units = 0;
    int64_t dp, sk_tiles, units;
    if (!stream_k_split(p->num_tiles, p->num_kb, pairs, tiles_per_item, &dp, &sk_tiles, &units)) return TGEMM_OK;
    const int64_t slots = units * kMaxSegments * tiles_per_item;    // one partial tile per slot
    const size_t part = (size_t)slots * kPairBM * kPairBN * sizeof(float);
    int devno = 0;
    cudaGetDevice(&devno);
    tgemm_status st = split_workspace(devno, stream_ptr, part, &p->counters, &p->partials);
    if (st != TGEMM_OK) return st;
    if (!encode_3d(&p->tma_ws, TGEMM_F32, p->partials, (uint64_t)kPairBN, (uint64_t)(slots * kPairBM),
                   (uint64_t)kPairBN, 1, 0, 32, 32))
        return TGEMM_ERR_CUDA;
    p->dp_tiles = (int32_t)dp;
    p->sk_tiles = (int32_t)sk_tiles;
    p->sk_units = (int32_t)units;
    return TGEMM_OK;
}

// K = 0 with a fused epilogue: D = act(beta * C_in + bias), elementwise.
template <int OUT>
__global__ void epilogue_only_kernel(const __grid_constant__ GemmParams p)
{
    const int64_t total = (int64_t)p.M * p.N;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(e / p.N);
        const int64_t n = e - (int64_t)m * p.N;
        float cin = 0.f;
        if (p.epi & 2) {
            const int64_t ci = (int64_t)m * p.ldc_in + n;
            if (OUT == OUT_F32) cin = static_cast<const float *>(p.cin_ptr)[ci];
            else if (OUT == OUT_F16) cin = __half2float(static_cast<const __half *>(p.cin_ptr)[ci]);
            else cin = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.cin_ptr)[ci]);
        }
        store_out<OUT>(p.c_ptr, (int64_t)m * p.ldc + n, epi_value(p, 0.f, cin, n));
    }
}

// Epilogue arguments: host checks and the kernel parameter fields.
tgemm_status epilogue_params(const tgemm_epilogue *ep, int64_t M, int64_t N, int out_dtype, GemmParams *p,
                             const Batch &bt = Batch())
{
    p->alpha = 1.f;
    p->beta = 0.f;
    p->epi = 0;
    if (!ep) return TGEMM_OK;
    if (ep->act != TGEMM_ACT_NONE && ep->act != TGEMM_ACT_RELU && ep->act != TGEMM_ACT_GELU_TANH)
        return TGEMM_ERR_INVALID_ARG;
    if (ep->bias && ep->bias_dtype != TGEMM_F16 && ep->bias_dtype != TGEMM_BF16 && ep->bias_dtype != TGEMM_F32)
        return TGEMM_ERR_INVALID_ARG;
    if (ep->bias && ((uintptr_t)ep->bias % 16) != 0) return TGEMM_ERR_MISALIGNED;   // read in 16-byte runs
    p->alpha = ep->alpha;
    p->beta = ep->beta;
    p->bias = ep->bias;
    p->bias_dtype = ep->bias_dtype;
    p->act = ep->act;
    const bool identity = ep->alpha == 1.f && ep->beta == 0.f && !ep->bias && ep->act == TGEMM_ACT_NONE;
    p->epi = identity ? 0 : 1;
    if (ep->beta != 0.f) {
        const size_t eo = elem_size(out_dtype);
        if (!ep->c_in || ep->ldc_in < N) return TGEMM_ERR_INVALID_ARG;
        if (((uintptr_t)ep->c_in % 16) != 0 || ((uint64_t)ep->ldc_in * eo) % 16 != 0) return TGEMM_ERR_MISALIGNED;
        p->epi |= 2;
        p->cin_ptr = ep->c_in;
        p->ldc_in = ep->ldc_in;
        // C_in steps through the batches like C (stride_c)
        if (M > 0 && N > 0 &&
            !encode_3d(&p->tma_cin, out_dtype, ep->c_in, (uint64_t)N, (uint64_t)M, (uint64_t)ep->ldc_in,
                       (uint64_t)bt.count, (uint64_t)(bt.count > 1 ? bt.sc : 0), (uint32_t)(128 / eo), 32))
            return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

// What one call launched, for the TGEMM_LOG trace (filled by the launch
// paths below, printed by run_impl's caller-facing wrapper).
struct LaunchRecord {
    const char *kernel = nullptr;   // nullptr: nothing launched
    tgemm_config cfg{};
    int grid = 0;                   // CTAs launched
    int dp_tiles = 0, sk_units = 0; // stream-K split (0 units: whole tiles)
};
thread_local LaunchRecord t_rec;

bool log_enabled()
{
    static const bool on = [] {
        const char *s = std::getenv("TGEMM_LOG");
        return s != nullptr && *s != '\0' && std::strcmp(s, "0") != 0;
    }();
    return on;
}

const char *dtype_name(int dt)
{
    switch (dt) {
    case TGEMM_F16: return "f16";
    case TGEMM_BF16: return "bf16";
    case TGEMM_F32: return "f32";
    case TGEMM_E4M3: return "e4m3";
    case TGEMM_E5M2: return "e5m2";
    }
    return "?";
}

// One stderr line per call when TGEMM_LOG is set (and not "0"): the problem,
// whether the configuration was the caller's or the library's choice, what
// was launched with which configuration, and the call's status.
void log_call(const char *entry, int64_t batch, int64_t M, int64_t N, int64_t K, int b_layout, int in_dtype,
              int out_dtype, bool forced, bool epilogue, tgemm_status st)
{
    const LaunchRecord &r = t_rec;
    char what[256];
    if (r.kernel)
        std::snprintf(what, sizeof what,
                      "%s bm=%d bn=%d bk=%d stages=%d cluster_m=%d group_m=%d split_k=%d swap_ab=%d grid=%d "
                      "dp_tiles=%d sk_units=%d",
                      r.kernel, r.cfg.bm, r.cfg.bn, r.cfg.bk, r.cfg.stages, r.cfg.cluster_m, r.cfg.group_m,
                      r.cfg.split_k, r.cfg.swap_ab, r.grid, r.dp_tiles, r.sk_units);
    else
        std::snprintf(what, sizeof what, "no kernel");
    std::fprintf(stderr, "tgemm: %s batch=%lld M=%lld N=%lld K=%lld B=%s in=%s out=%s epilogue=%d config=%s -> %s; %s\n",
                 entry, (long long)batch, (long long)M, (long long)N, (long long)K,
                 b_layout == TGEMM_B_KN ? "KxN" : "NxK", dtype_name(in_dtype), dtype_name(out_dtype),
                 epilogue ? 1 : 0, forced ? "caller" : "library", what, tgemm_status_string(st));
}

// C^T = B^T A^T on a swap-AB split-K kernel (M <= 64, or M <= 128 in-cluster): the workspace
// reduction (swap_ab = 1) or the in-cluster one (swap_ab = 2).
tgemm_status run_skinny(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                        int b_layout, void *C, int64_t ldc, int in_dtype, int out_dtype, void *stream_ptr,
                        const tgemm_config &cfg, const KernelVariant *var, DeviceState *dev,
                        const tgemm_epilogue *ep)
{
    const bool w_mn = b_layout == TGEMM_B_KN;
    const int npad = cfg.bn;
    const int64_t tiles_n = ceil_div(N, kSkinnyRows);
    int splits = cfg.split_k;
    if (cfg.swap_ab == 1 && tiles_n > kMaxSkinnyTiles) splits = 1;
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    // K elements per 128-byte k-block row: 64 for FP16/BF16, 128 for FP8
    const uint32_t kbe = (uint32_t)kblock_elems(in_dtype);
    bool ok = encode_2d(&p.tma_a, in_dtype, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, kbe, (uint32_t)npad);
    if (w_mn)
        ok = ok && encode_2d(&p.tma_b, in_dtype, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, 64, kBK);
    else
        ok = ok && encode_2d(&p.tma_b, in_dtype, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, kbe, kSkinnyRows);
    if (!ok) return TGEMM_ERR_CUDA;
    p.M = (int32_t)M;
    p.N = (int32_t)N;
    p.K = (int32_t)K;
    p.tiles_m = 1;
    p.tiles_n = (int32_t)tiles_n;
    p.num_tiles = (int32_t)tiles_n;
    p.num_kb = (int32_t)ceil_div(K, (int64_t)kbe);
    p.group_m = 1;
    p.idesc = make_idesc(mma_type(in_dtype), false, kSkinnyRows, npad, w_mn);
    p.status = dev->status;
    p.clock_rec = dev->clock_rec.load(std::memory_order_relaxed);
    p.timeout_ns = wait_timeout_ns();
    p.c_ptr = C;
    p.ldc = ldc;
    p.splits = splits;
    if (cfg.swap_ab == 2) {
        // Dependent-launch overlap of the in-cluster kernel: when the next
        // launch's CTAs fit beside this one's (a grid of at most one CTA per
        // SM) or each CTA streams a long slice (at least 12 k-blocks), start
        // the next launch once every CTA has issued its last load and let it
        // prefetch its whole weight slice; otherwise start it at once with a
        // short prefetch.  Measured on one GB300, graph-replayed, best
        // configuration per shape: 16x4096x4096 8.9 -> 8.2 us, 64x4096x4096
        // 11.5 -> 11.0, 32x4096x8192 14.9 -> 14.4, 16x14336x4096 20.8 -> 19.9;
        // 16x16384x1024 (256 CTAs of 8 k-blocks) stays early, 7.5 against 8.0.
        const int64_t kb_per_cta = ceil_div(ceil_div(K, (int64_t)kbe), splits);
        p.late_trigger = (kb_per_cta >= 12 || tiles_n * splits <= dev->sm_count) ? 1 : 0;
        p.prefetch_kb = p.late_trigger ? (int32_t)kb_per_cta : kSkinnyPrefetchKb;
    }
    tgemm_status est = epilogue_params(ep, M, N, out_dtype, &p);
    if (est != TGEMM_OK) return est;
    if (splits > 1 && cfg.swap_ab == 1) {
        int devno = 0;
        cudaGetDevice(&devno);
        const size_t part = (size_t)splits * (size_t)tiles_n * (size_t)npad * kSkinnyRows * sizeof(float);
        tgemm_status st = split_workspace(devno, stream_ptr, part, &p.counters, &p.partials);
        if (st != TGEMM_OK) return st;
    }
    const int64_t grid = tiles_n * splits;
    if (grid > INT32_MAX) return TGEMM_ERR_UNSUPPORTED;
    t_rec.kernel = cfg.swap_ab == 2 ? "skinny-cluster-splitk" : "skinny-workspace-splitk";
    t_rec.cfg = cfg;
    t_rec.cfg.split_k = splits;
    t_rec.grid = (int)grid;
    if (var->launch(p, (int)grid, static_cast<cudaStream_t>(stream_ptr)) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

// Rows of A or B whose pitch is not a multiple of 128 bytes make every
// 128-byte TMA box row straddle two cache lines: about three times the L2
// requests per byte (measured: 19.5 M against 6.6 M on 4096 x 3072 x 5000).
// The quad kernel fetches each A half-tile once for two pairs, a quarter
// fewer requests, and measured 17-20 % faster than the pair kernel on such
// shapes (110 -> 91 us on 4000 x 3000 x 5000); on aligned rows the pair
// kernel's independent rings win.  So a pair choice (whole tiles or
// stream-K) becomes a quad one when rows are misaligned.
void prefer_quad_for_misaligned_rows(tgemm_config *cfg, int64_t M, int64_t N, int64_t lda, int64_t ldb,
                                     int in_dtype, int sm_count, bool batched = false)
{
    if (cfg->cluster_m != 2 || cfg->swap_ab != 0) return;
    const int64_t e = (int64_t)elem_size(in_dtype);
    if ((lda * e) % 128 == 0 && (ldb * e) % 128 == 0) return;
    if (M < 256 || N < 512) return;
    cfg->cluster_m = 4;
    // stream-K where a leftover wave is at most half full (plan_stream_k
    // keeps whole blocks otherwise): 2000 x 3000 x 5000 53.9 -> 44.0 us
    cfg->split_k = batched ? 1 : 0;
    cfg->group_m = 8;
    cfg->grid = quad_grid(M, N, cfg->split_k, sm_count);
}

// GROUP_SIZE_M of the grouped order from the L2 footprint it implies.  A
// band of group_m tile rows that spans several waves of resident tiles reads
// all of B once, and its A rows again in every wave; they stay in L2 only
// while they, the B columns of about two waves and one wave's C tiles fit in
// what L2 keeps for them.  Fewer, taller bands read B fewer times.  Measured
// with ncu (DRAM bytes per launch, pair kernel): 8192^3 FP16 2.87x the
// algorithmic bytes at group 8 or 10, 2.56x at 12, 2.86x at 14 (bands 14,
// 14, 4: the short last band reads B once more); 16384 x 14336 x 4096 BF16
// 2.23x at 8, 1.75x at 16 and 1.97x at 24.  This footprint model with a
// 64 MiB budget picks 16 there; for 8192^3 no band fits and the smallest
// footprint, bands of 11, 11 and 10 rows, is taken.  An LRU model of the
// schedule (l2_schedule_model.py: a 64 MiB cache, each wave's pairs in
// lockstep over k, which ranks the measured heights as ncu did) puts this
// choice within 1 % of its best height in DRAM reads on 44 of 48 shapes
// from 8192 to 24576 rows and columns and K 4096-16384, at most 4.6 % above
// it (8192^3, where 12 is best), and above a group of 8 on two shapes, by at
// most 1.1 %.  The tutorial's group of
// 8 stays where A and B together are small enough to stay in L2 (4000 x 3000
// x 5000 reads about its algorithmic bytes at group 8) and where a band of 8
// rows holds less than two waves (there a wave spans bands and B, not A, is
// what the next wave re-reads).
constexpr double kL2BandBudget = 64.0 * 1024 * 1024;
constexpr double kL2OperandsFit = 96.0 * 1024 * 1024;

int l2_group_m(int64_t M, int64_t N, int64_t K, int bm, int unit_bn, int in_dtype, int out_dtype, int64_t resident)
{
    const int64_t tm = ceil_div(M, bm), tn = ceil_div(N, unit_bn);
    const double e = (double)elem_size(in_dtype), eo = (double)elem_size(out_dtype);
    const double row = (double)bm * (double)K * e, col = (double)unit_bn * (double)K * e;
    if (resident < 1 || (double)tm * row + (double)tn * col <= kL2OperandsFit) return kDefaultGroupM;
    if ((int64_t)kDefaultGroupM * tn < 2 * resident) return kDefaultGroupM;
    const double c_wave = (double)resident * bm * unit_bn * eo;
    int64_t best_gm = kDefaultGroupM, prev_gm = 0;
    double best = 0;
    for (int64_t nb = 1; nb <= tm; ++nb) {
        const int64_t gm = ceil_div(tm, nb);                 // bands of near-equal height
        if (gm == prev_gm) continue;
        prev_gm = gm;
        if (gm * tn < 2 * resident) break;                   // later bands are shorter still
        // B columns a wave spans, counted fractionally: rounding up to whole
        // columns made several heights tie (16, 12 and 10 on 48 tile rows)
        const double cols = std::min((double)tn, (double)resident / (double)gm);
        const double f = (double)gm * row + 2.0 * cols * col + c_wave;
        if (f <= kL2BandBudget) return (int)gm;              // the fewest bands that fit
        if (best == 0 || f < best) {
            best = f;
            best_gm = gm;
        }
    }
    return (int)best_gm;
}

// The group for an automatically chosen tile configuration (single
// problems; strided batches keep the default).  The picker table measured
// groups of 8 and 16 for the pair kernel's whole tiles in the power-capped
// steady state, and where 16 won it stays (also on shapes whose operands fit
// in L2, where the model has no say); the model only makes a default group
// of 8 taller.  On 8192^3 FP16 (pair, stream-K tail) that is 11: DRAM bytes
// 2.77x -> 2.69x the algorithmic ones, per-clock tensor efficiency 0.959 ->
// 0.966 in a 50-launch burst; on 8192^3 TF32 (quad) 11, within noise.
void l2_group_config(tgemm_config *cfg, int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype,
                     int sm_count)
{
    if (cfg->swap_ab || cfg->group_m != kDefaultGroupM) return;
    int64_t resident;
    int unit_bn = cfg->bn;
    if (cfg->cluster_m == 2) {
        resident = sm_count / 2;
    } else if (cfg->cluster_m == 4) {
        resident = sm_count / 4;
        unit_bn = 2 * cfg->bn;                                // a quad's block is two pair tiles wide
    } else {
        resident = (int64_t)sm_count * tile_ctas_per_sm(cfg->bn, cfg->stages);
    }
    const int g = l2_group_m(M, N, K, cfg->bm, unit_bn, in_dtype, out_dtype, resident);
    if (g > cfg->group_m) cfg->group_m = g;
}

tgemm_status run_body(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                      int64_t ldb, int b_layout, void *C, int64_t ldc, int in_dtype, int out_dtype,
                      void *stream_ptr, const tgemm_config *forced, const tgemm_epilogue *ep,
                      const Batch &bt)
{
    bool noop = false;
    tgemm_status st = validate(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, &noop);
    if (st != TGEMM_OK) return st;
    tgemm_config cfg;
    const KernelVariant *var = nullptr;
    if (forced) {
        cfg = *forced;
        st = legal_config(cfg, M, K, out_dtype, b_layout, &var, in_dtype);
        if (st != TGEMM_OK) return st;
        if (bt.count > 1 && cfg.swap_ab) return TGEMM_ERR_UNSUPPORTED;   // the skinny kernels are not batched
    }
    if (noop || bt.count == 0) return TGEMM_OK;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TGEMM_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    const size_t eo = elem_size(out_dtype);
    {
        // epilogue arguments are checked before anything is launched
        GemmParams probe;
        std::memset(&probe, 0, sizeof probe);
        tgemm_status est = epilogue_params(ep, 0, N, out_dtype, &probe);
        if (est != TGEMM_OK) return est;
        if (K == 0 && probe.epi) {
            // The empty sum under the epilogue: D = act(beta * C_in + bias), per batch.
            for (int64_t b = 0; b < bt.count; ++b) {
                GemmParams q;
                std::memset(&q, 0, sizeof q);
                epilogue_params(ep, 0, N, out_dtype, &q);
                q.M = (int32_t)M;
                q.N = (int32_t)N;
                q.c_ptr = static_cast<char *>(C) + (size_t)(b * bt.sc) * eo;
                q.ldc = ldc;
                if (q.epi & 2) q.cin_ptr = static_cast<const char *>(q.cin_ptr) + (size_t)(b * bt.sc) * eo;
                const int64_t total = M * N;
                const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4 * (int64_t)dev->sm_count);
                t_rec.kernel = "epilogue-only";
                t_rec.grid = blocks;
                if (out_dtype == TGEMM_F32) epilogue_only_kernel<OUT_F32><<<blocks, 256, 0, stream>>>(q);
                else if (out_dtype == TGEMM_F16) epilogue_only_kernel<OUT_F16><<<blocks, 256, 0, stream>>>(q);
                else epilogue_only_kernel<OUT_BF16><<<blocks, 256, 0, stream>>>(q);
                if (cudaGetLastError() != cudaSuccess) return TGEMM_ERR_CUDA;
            }
            return TGEMM_OK;
        }
    }
    if (K == 0) {
        // The empty sum: C = 0 (all-zero bits are +0 in every output type).
        t_rec.kernel = "memset";
        for (int64_t b = 0; b < bt.count; ++b)
            if (cudaMemset2DAsync(static_cast<char *>(C) + (size_t)(b * bt.sc) * eo, (size_t)ldc * eo, 0,
                                  (size_t)N * eo, (size_t)M, stream) != cudaSuccess) {
                cudaGetLastError();
                return TGEMM_ERR_CUDA;
            }
        return TGEMM_OK;
    }
    if (!forced) {
        choose_config(M, N, K, b_layout, pick_class(in_dtype), dev->sm_count, &cfg);
        if (bt.count > 1) {
            // The table was measured on single problems and the skinny kernels
            // are not batched: the wave model over the tiles of all batches.
            choose_config_model(M, N, K, dev->sm_count, &cfg, bt.count, false, pick_class(in_dtype));
        }
        if (!swap_supported(in_dtype, cfg.swap_ab)) {
            // a table entry of another operand class: the tile kernels
            choose_config_model(M, N, K, dev->sm_count, &cfg, bt.count, false, pick_class(in_dtype));
        }
        if (bt.count > 1 && cfg.split_k == 0) cfg.split_k = 1;   // many batches fill the waves themselves
        prefer_quad_for_misaligned_rows(&cfg, M, N, lda, ldb, in_dtype, dev->sm_count, bt.count > 1);
        if (bt.count == 1) l2_group_config(&cfg, M, N, K, in_dtype, out_dtype, dev->sm_count);
        cfg.grid = 0;   // sized below from the tiles of all batches
        st = legal_config(cfg, M, K, out_dtype, b_layout, &var, in_dtype);
        if (st != TGEMM_OK) return st;
    }
    if (cfg.swap_ab)
        return run_skinny(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream_ptr, cfg, var,
                          dev, ep);
    const bool b_mn = b_layout == TGEMM_B_KN;
    const bool pair = cfg.cluster_m == 2;
    const bool quad = cfg.cluster_m == 4;
    // a quad's unit of work is a 256 x 512 block (two pair tiles side by side)
    const TileGrid grid(M, N, cfg.bm, quad ? 2 * cfg.bn : cfg.bn);
    // Rows of A and columns of B one CTA stages (loads) per k-block.
    const uint32_t b_box_rows = (pair || quad) ? (uint32_t)(cfg.bn / 2) : (uint32_t)cfg.bn;
    const uint32_t a_box_rows = quad ? (uint32_t)(kBM / 2) : (uint32_t)kBM;

    GemmParams p;
    std::memset(&p, 0, sizeof p);
    const uint64_t nb = (uint64_t)bt.count;
    const uint64_t sa = bt.count > 1 ? (uint64_t)bt.sa : 0, sb = bt.count > 1 ? (uint64_t)bt.sb : 0;
    const uint64_t sc = bt.count > 1 ? (uint64_t)bt.sc : 0;
    const uint32_t kbe = (uint32_t)kblock_elems(in_dtype);   // K elements per 128-byte k-block row
    bool ok = encode_3d(&p.tma_a, in_dtype, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, nb, sa, kbe, a_box_rows);
    if (b_mn)
        ok = ok && encode_3d(&p.tma_b, in_dtype, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, nb, sb, 64, kBK);
    else
        ok = ok && encode_3d(&p.tma_b, in_dtype, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, nb, sb, kbe,
                             b_box_rows);
    ok = ok && encode_3d(&p.tma_c, out_dtype, C, (uint64_t)N, (uint64_t)M, (uint64_t)ldc, nb, sc,
                         (uint32_t)(128 / eo), 32);
    if (!ok) return TGEMM_ERR_CUDA;
    if (grid.count() * bt.count >= ((int64_t)1 << 31)) return TGEMM_ERR_UNSUPPORTED;
    // the kernels map tiles with 32-bit arithmetic (grouped_tile32)
    if ((int64_t)cfg.group_m * grid.tiles_n >= ((int64_t)1 << 31)) return TGEMM_ERR_UNSUPPORTED;
    p.M = (int32_t)M;
    p.N = (int32_t)N;
    p.K = (int32_t)K;
    p.tiles_m = (int32_t)grid.tiles_m;
    p.tiles_n = (int32_t)grid.tiles_n;
    p.tiles_per_batch = (int32_t)grid.count();
    p.a_batched = sa != 0;
    p.b_batched = sb != 0;
    p.num_tiles = (int32_t)(grid.count() * bt.count);
    p.num_kb = (int32_t)ceil_div(K, kbe);
    p.group_m = cfg.group_m;
    // kind::f16: type codes 0 F16 / 1 BF16; kind::f8f6f4: 0 E4M3 / 1 E5M2
    p.idesc = make_idesc(mma_type(in_dtype), b_mn, cfg.bm, cfg.bn);
    p.status = dev->status;
    p.clock_rec = dev->clock_rec.load(std::memory_order_relaxed);
    p.timeout_ns = wait_timeout_ns();
    // Odd waves of whole tiles run their K loop backwards (work_kb in the pair
    // kernel): on 8192^3 FP16 the pair kernel's DRAM reads fell from 1.146 to
    // 1.024 GB per launch (GROUP_SIZE_M 8) and from 1.237 to 0.983 GB (16),
    // worth 0.4-2.6 % in the power-capped steady state; no change on the
    // quad's misaligned 4000 x 3000 x 5000 or on 16384 x 14336 x 4096.
    p.k_alternate = 1;
    st = epilogue_params(ep, M, N, out_dtype, &p, bt);
    if (st != TGEMM_OK) return st;

    int g;
    p.dp_tiles = p.num_tiles;
    if (pair) {
        // grid counts CTAs: an even number, at most two per tile and two per
        // resident pair
        int pairs = cfg.grid > 0 ? cfg.grid / 2 : dev->sm_count / 2;
        const int resident = resident_pairs(dev, var);
        if (pairs > resident) pairs = resident;
        if (cfg.split_k != 0 && pairs > p.num_tiles) pairs = p.num_tiles;
        if (pairs < 1) pairs = 1;
        g = 2 * pairs;
        if (cfg.split_k == 0) {
            tgemm_status st2 = plan_stream_k(&p, pairs, dev, stream_ptr);
            if (st2 != TGEMM_OK) return st2;
            if (p.sk_units == 0 && pairs > p.num_tiles) g = 2 * p.num_tiles;
            if (p.sk_units > 0 && p.dp_tiles == 0) g = 2 * p.sk_units;   // only the sharing pairs have work
        }
    } else if (quad) {
        // grid counts CTAs: four per quad, at most one quad per block with
        // whole blocks
        int quads = cfg.grid > 0 ? cfg.grid / 4 : dev->sm_count / 4;
        const int resident = resident_pairs(dev, var);       // resident quads for this variant
        if (quads > resident) quads = resident;
        if (cfg.split_k != 0 && quads > p.num_tiles) quads = p.num_tiles;
        if (quads < 1) quads = 1;
        g = 4 * quads;
        if (cfg.split_k == 0) {
            tgemm_status st2 = plan_stream_k(&p, quads, dev, stream_ptr, 2);
            if (st2 != TGEMM_OK) return st2;
            if (p.sk_units == 0 && quads > p.num_tiles) g = 4 * p.num_tiles;
            if (p.sk_units > 0 && p.dp_tiles == 0) g = 4 * p.sk_units;   // only the sharing quads have work
        }
    } else {
        g = cfg.grid > 0 ? cfg.grid : dev->sm_count * tile_ctas_per_sm(cfg.bn, cfg.stages);
        if (g > p.num_tiles) g = p.num_tiles;
        if (g < 1) g = 1;
    }
    t_rec.kernel = pair ? "pair" : quad ? "quad" : "tile";
    t_rec.cfg = cfg;
    t_rec.grid = g;
    t_rec.dp_tiles = p.dp_tiles;
    t_rec.sk_units = p.sk_units;
    if (var->launch(p, g, stream) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

tgemm_status run_impl(const char *entry, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                      const void *B, int64_t ldb, int b_layout, void *C, int64_t ldc, int in_dtype, int out_dtype,
                      void *stream_ptr, const tgemm_config *forced, const tgemm_epilogue *ep = nullptr,
                      const Batch &bt = Batch())
{
    t_rec = LaunchRecord();
    const tgemm_status st = run_body(M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream_ptr,
                                     forced, ep, bt);
    if (log_enabled()) log_call(entry, bt.count, M, N, K, b_layout, in_dtype, out_dtype, forced != nullptr,
                                ep != nullptr, st);
    return st;
}

}  // namespace
}  // namespace tgemm

using namespace tgemm;

TGEMM_EXPORT tgemm_status tgemm_run(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                                    const void *B, int64_t ldb, tgemm_b_layout b_layout, void *C,
                                    int64_t ldc, tgemm_dtype in_dtype, tgemm_dtype out_dtype, void *stream)
{
    return run_impl("tgemm_run", M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream, nullptr);
}

TGEMM_EXPORT tgemm_status tgemm_run_config(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                                           const void *B, int64_t ldb, tgemm_b_layout b_layout, void *C,
                                           int64_t ldc, tgemm_dtype in_dtype, tgemm_dtype out_dtype,
                                           void *stream, const tgemm_config *cfg)
{
    if (!cfg) return TGEMM_ERR_INVALID_ARG;
    return run_impl("tgemm_run_config", M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream, cfg);
}

TGEMM_EXPORT tgemm_status tgemm_run_ex(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                                       int64_t ldb, tgemm_b_layout b_layout, void *C, int64_t ldc,
                                       tgemm_dtype in_dtype, tgemm_dtype out_dtype, void *stream,
                                       const tgemm_epilogue *ep, const tgemm_config *cfg)
{
    return run_impl("tgemm_run_ex", M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype, stream, cfg,
                    ep);
}

TGEMM_EXPORT tgemm_status tgemm_run_strided_batched(int64_t batch, int64_t M, int64_t N, int64_t K, const void *A,
                                                    int64_t lda, int64_t stride_a, const void *B, int64_t ldb,
                                                    int64_t stride_b, tgemm_b_layout b_layout, void *C, int64_t ldc,
                                                    int64_t stride_c, tgemm_dtype in_dtype, tgemm_dtype out_dtype,
                                                    void *stream, const tgemm_epilogue *ep, const tgemm_config *cfg)
{
    if (batch < 0 || stride_a < 0 || stride_b < 0 || stride_c < 0) return TGEMM_ERR_INVALID_ARG;
    if (batch > 1 && M > 0 && N > 0) {
        // Batches may share A or B (stride 0) but must not overlap otherwise;
        // outputs never overlap.  Strides keep rows 16-byte aligned.
        const int64_t b_rows = b_layout == TGEMM_B_KN ? K : N;
        if ((stride_a != 0 && stride_a < M * lda) || (stride_b != 0 && stride_b < b_rows * ldb) ||
            stride_c < M * ldc)
            return TGEMM_ERR_INVALID_ARG;
        const size_t ei = elem_size(in_dtype), eo = elem_size(out_dtype);
        if (((uint64_t)stride_a * ei) % 16 || ((uint64_t)stride_b * ei) % 16 || ((uint64_t)stride_c * eo) % 16)
            return TGEMM_ERR_MISALIGNED;
        if (batch >= ((int64_t)1 << 31)) return TGEMM_ERR_UNSUPPORTED;
    }
    Batch bt;
    bt.count = batch;
    bt.sa = stride_a;
    bt.sb = stride_b;
    bt.sc = stride_c;
    return run_impl("tgemm_run_strided_batched", M, N, K, A, lda, B, ldb, b_layout, C, ldc, in_dtype, out_dtype,
                    stream, cfg, ep, bt);
}

namespace tgemm {
namespace {

tgemm_status query_args(int64_t M, int64_t N, int64_t K, int b_layout, int in_dtype, int out_dtype,
                        const tgemm_config *out_cfg)
{
    if (!out_cfg) return TGEMM_ERR_INVALID_ARG;
    if (b_layout != TGEMM_B_KN && b_layout != TGEMM_B_NK) return TGEMM_ERR_INVALID_ARG;
    if (in_dtype != TGEMM_F16 && in_dtype != TGEMM_BF16 && !tile_only(in_dtype)) return TGEMM_ERR_INVALID_ARG;
    if (tile_only(in_dtype) && b_layout != TGEMM_B_NK) return TGEMM_ERR_UNSUPPORTED;
    if (out_dtype != TGEMM_F16 && out_dtype != TGEMM_BF16 && out_dtype != TGEMM_F32)
        return TGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_ARG;
    return TGEMM_OK;
}

// The configuration tgemm_run chooses for a single problem with tightly
// packed rows (lda = K, ldb = K for N x K or N for K x N) on a GPU with
// sm_count SMs: the same steps as its own choice, in the same order.
void auto_config(int64_t M, int64_t N, int64_t K, int b_layout, int in_dtype, int out_dtype, int sm_count,
                 tgemm_config *cfg)
{
    choose_config(M > 0 ? M : 1, N > 0 ? N : 1, K > 0 ? K : 1, b_layout, pick_class(in_dtype), sm_count, cfg);
    if (!swap_supported(in_dtype, cfg->swap_ab))
        choose_config_model(M > 0 ? M : 1, N, K, sm_count, cfg, 1, false, pick_class(in_dtype));
    prefer_quad_for_misaligned_rows(cfg, M, N, K, b_layout == TGEMM_B_KN ? N : K, in_dtype, sm_count);
    l2_group_config(cfg, M > 0 ? M : 1, N > 0 ? N : 1, K > 0 ? K : 1, in_dtype, out_dtype, sm_count);
}

}  // namespace
}  // namespace tgemm

TGEMM_EXPORT tgemm_status tgemm_query_config(int64_t M, int64_t N, int64_t K, tgemm_b_layout b_layout,
                                             tgemm_dtype in_dtype, tgemm_dtype out_dtype,
                                             tgemm_config *out_cfg)
{
    tgemm_status st = query_args(M, N, K, b_layout, in_dtype, out_dtype, out_cfg);
    if (st != TGEMM_OK) return st;
    DeviceState *dev = nullptr;
    st = device_state(&dev);
    if (st != TGEMM_OK) return st;
    auto_config(M, N, K, b_layout, in_dtype, out_dtype, dev->sm_count, out_cfg);
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_query_config_sms(int64_t M, int64_t N, int64_t K, tgemm_b_layout b_layout,
                                                 tgemm_dtype in_dtype, tgemm_dtype out_dtype, int sm_count,
                                                 tgemm_config *out_cfg)
{
    tgemm_status st = query_args(M, N, K, b_layout, in_dtype, out_dtype, out_cfg);
    if (st != TGEMM_OK) return st;
    if (sm_count < 1 || sm_count > 4096) return TGEMM_ERR_INVALID_ARG;
    auto_config(M, N, K, b_layout, in_dtype, out_dtype, sm_count, out_cfg);
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_check(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    uint32_t *status = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        status = g_dev[dev].status;
    }
    // The library's status word and the allocation-free path's (which lives
    // in that path's built-in array); either may not exist yet.
    uint32_t first = 0;
    uint32_t *words[2] = {status, noalloc_status_word(dev)};
    for (uint32_t *w : words) {
        if (!w) continue;
        uint32_t word = 0;
        if (cudaMemcpy(&word, w, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        if (word == 0) continue;
        if (first == 0) first = word;
        if (cudaMemset(w, 0, sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
    }
    if (first == 0) return TGEMM_OK;
    g_last_fault.store(first);
    {
        // A kernel gave up part-way: split-K arrival counters may be left
        // non-zero; clear them so the next call starts clean.  (The
        // allocation-free path clears its counters before every launch.)
        std::lock_guard<std::mutex> lk(g_mu);
        for (auto &kv : g_ws)
            if (kv.first.first == dev && kv.second.ptr) cudaMemset(kv.second.ptr, 0, kCounterBytes);
    }
    return (first >> 28) == kFaultTimeout ? TGEMM_ERR_TIMEOUT : TGEMM_ERR_CUDA;
}

TGEMM_EXPORT uint32_t tgemm_last_fault_code(void) { return g_last_fault.load(); }

TGEMM_EXPORT const char *tgemm_status_string(tgemm_status s)
{
    switch (s) {
    case TGEMM_OK: return "ok";
    case TGEMM_ERR_INVALID_ARG: return "invalid argument (negative size, NULL pointer, short leading dimension or bad enum)";
    case TGEMM_ERR_UNSUPPORTED: return "unsupported dtype, size or configuration";
    case TGEMM_ERR_MISALIGNED: return "pointer or leading dimension not 16-byte aligned";
    case TGEMM_ERR_ARCH: return "current device is not sm_103 (GB300)";
    case TGEMM_ERR_CUDA: return "CUDA runtime or driver error";
    case TGEMM_ERR_OOM: return "out of device memory for library workspace";
    case TGEMM_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    }
    return "unknown status";
}

TGEMM_EXPORT void tgemm_shutdown(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = -1;
    cudaGetDevice(&cur);
    for (auto &kv : g_ws) {
        if (kv.second.ptr) {
            cudaSetDevice(kv.first.first);
            cudaFree(kv.second.ptr);
        }
    }
    g_ws.clear();
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_dev[d].status) {
            cudaSetDevice(d);
            cudaFree(g_dev[d].status);
        }
        g_dev[d].ready = false;
        g_dev[d].sm_count = g_dev[d].cc_major = g_dev[d].cc_minor = 0;
        g_dev[d].status = nullptr;
        g_dev[d].pairs.clear();
        g_dev[d].clock_rec.store(nullptr);
    }
    if (cur >= 0) cudaSetDevice(cur);
    cudaGetLastError();
}

TGEMM_EXPORT tgemm_status tgemm_tile_coord(int64_t M, int64_t N, int bm, int bn, int group_m, int64_t bid,
                                           int64_t *bid_m, int64_t *bid_n)
{
    if (M <= 0 || N <= 0 || bm <= 0 || bn <= 0 || group_m <= 0 || !bid_m || !bid_n)
        return TGEMM_ERR_INVALID_ARG;
    const TileGrid g(M, N, bm, bn);
    if (bid < 0 || bid >= g.count()) return TGEMM_ERR_INVALID_ARG;
    if (g.count() * (int64_t)group_m < ((int64_t)1 << 31)) {
        // the kernels' 32-bit form (every grid they run fits it)
        int32_t r, c;
        grouped_tile32((int32_t)g.tiles_m, (int32_t)g.tiles_n, group_m, (int32_t)bid, r, c);
        *bid_m = r;
        *bid_n = c;
    } else {
        grouped_tile(g.tiles_m, g.tiles_n, group_m, bid, *bid_m, *bid_n);
    }
    return TGEMM_OK;
}

namespace tgemm {
// tgemm_debug.cu
cudaError_t launch_tile_order_probe(int32_t tiles_m, int32_t tiles_n, int32_t group_m, int32_t count, int32_t *rows,
                                    int32_t *cols, cudaStream_t st);
}  // namespace tgemm

TGEMM_EXPORT tgemm_status tgemm_group_size(int64_t M, int64_t N, int64_t K, int bm, int unit_bn, int in_dtype,
                                           int out_dtype, int resident, int *group_m)
{
    if (M < 1 || N < 1 || K < 1 || bm < 1 || unit_bn < 1 || resident < 1 || !group_m) return TGEMM_ERR_INVALID_ARG;
    if (in_dtype < TGEMM_F16 || in_dtype > TGEMM_E5M2 || out_dtype < TGEMM_F16 || out_dtype > TGEMM_F32)
        return TGEMM_ERR_INVALID_ARG;
    *group_m = l2_group_m(M, N, K, bm, unit_bn, in_dtype, out_dtype, resident);
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_stream_k_plan(int64_t items, int64_t k_blocks, int units, int tiles_per_item,
                                              int64_t *dp_items, int64_t *sk_items, int64_t *sk_units)
{
    if (items < 0 || k_blocks < 1 || units < 1 || (tiles_per_item != 1 && tiles_per_item != 2) || !dp_items ||
        !sk_items || !sk_units)
        return TGEMM_ERR_INVALID_ARG;
    int64_t dp = items, sk = 0, u = 0;
    if (!stream_k_split(items, k_blocks, units, tiles_per_item, &dp, &sk, &u)) {
        dp = items;
        sk = 0;
        u = 0;
    }
    *dp_items = dp;
    *sk_items = sk;
    *sk_units = u;
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_debug_tile_order(int64_t M, int64_t N, int bm, int bn, int group_m, int32_t *rows,
                                                 int32_t *cols, void *stream)
{
    if (M <= 0 || N <= 0 || bm <= 0 || bn <= 0 || group_m <= 0 || !rows || !cols) return TGEMM_ERR_INVALID_ARG;
    const TileGrid g(M, N, bm, bn);
    // the kernels' 32-bit form: the host keeps every grid they run below this
    if (g.count() * (int64_t)group_m >= ((int64_t)1 << 31)) return TGEMM_ERR_UNSUPPORTED;
    DeviceState *dev = nullptr;
    tgemm_status st = device_state(&dev);
    if (st != TGEMM_OK) return st;
    if (launch_tile_order_probe((int32_t)g.tiles_m, (int32_t)g.tiles_n, group_m, (int32_t)g.count(), rows, cols,
                                static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_debug_wait_timeout(uint32_t timeout_us, void *stream)
{
    DeviceState *dev = nullptr;
    tgemm_status st = device_state(&dev);
    if (st != TGEMM_OK) return st;
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return TGEMM_ERR_INVALID_ARG;
    if (launch_wait_timeout_probe(dev->status, (uint64_t)timeout_us * 1000ull,
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_debug_sm_clock(uint64_t *out, uint32_t duration_us, void *stream)
{
    if (!out || duration_us == 0 || duration_us > 100u * 1000u) return TGEMM_ERR_INVALID_ARG;
    if (((uintptr_t)out % 8) != 0) return TGEMM_ERR_MISALIGNED;
    DeviceState *dev = nullptr;
    tgemm_status st = device_state(&dev);
    if (st != TGEMM_OK) return st;
    if (launch_sm_clock_probe(out, (uint64_t)duration_us * 1000ull, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

TGEMM_EXPORT tgemm_status tgemm_debug_clock_record(uint64_t *rec)
{
    if (((uintptr_t)rec % 8) != 0) return TGEMM_ERR_MISALIGNED;
    DeviceState *dev = nullptr;
    tgemm_status st = device_state(&dev);
    if (st != TGEMM_OK) return st;
    dev->clock_rec.store(rec, std::memory_order_relaxed);
    return TGEMM_OK;
}
