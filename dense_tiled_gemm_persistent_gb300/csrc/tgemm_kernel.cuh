// Persistent, warp-specialised tcgen05 GEMM for sm_103a: C = A * B.
//
// The dataflow is the tile lifecycle the pages describe (load a BM x BK tile
// of A and a BK x BN tile of B, multiply-accumulate over the K loop, cast and
// write back; the double-buffered prefetch of the wmrh.cn essay "the parallel
// secret of a CUDA tile", section 2.2; the producer/consumer ring with full
// and empty events of the Croqtile tutorial's "Kernel 3: warp
// specialisation"), rebuilt on Blackwell hardware:
//
//   warp 0  producer  one thread issues TMA loads of A and B k-blocks into a
//                     STAGES-deep shared-memory ring (128-byte swizzle) and
//                     arms the stage's "full" mbarrier with the byte count;
//   warp 1  MMA       one thread waits on "full", issues BK/16 tcgen05.mma
//                     (M = 128, N = BN, K = 16) into an FP32 accumulator in
//                     tensor memory, and commits the stage back to "empty";
//                     after the last k-block it commits "tmem_full";
//   warps 2-5 epilogue  wait "tmem_full", read the accumulator with
//                     tcgen05.ld (warp w owns TMEM lanes 32*(w%4)..+31, i.e.
//                     tile rows), release the buffer ("tmem_empty"), cast
//                     FP32 -> output type with round-to-nearest-even, stage
//                     128-byte rows in swizzled shared memory and write them
//                     with TMA stores, which drop out-of-range rows/columns.
//
// Two accumulator buffers in tensor memory let the epilogue of tile i run
// while the MMAs of tile i+1 proceed.  The CTA loops over tiles
// bid = blockIdx.x, blockIdx.x + gridDim.x, ... in the grouped order of
// tgemm_sched.h, so the grid is one CTA per SM.
//
// Tails follow the CUDA Programming Guide 13.4.2 (unofficial Chinese
// translation), section 2.4.9.1: ceil(K/BK) k-blocks with the partial block
// zero-filled (TMA fills out-of-range elements with zeros), and partial M/N
// tiles clipped at the store.  A store whose box would start past the end of
// C is not issued at all.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <string.h>

#include "tgemm_params.h"
#include "tgemm_ptx.cuh"
#include "tgemm_sched.h"
#include "tgemm_wait.cuh"

namespace tgemm {

constexpr int kBM = 128;           // rows of one CTA tile = TMEM lanes
constexpr int kBK = 64;            // K depth of one stage: 64 x 2 bytes = one 128-byte swizzle row
constexpr int kUmmaK = 16;         // K of one tcgen05.mma kind::f16
// Operand kinds.  FP8 and TF32 operands keep the 16-bit byte geometry: a
// 128-byte row holds 128 FP8 or 32 FP32 elements and one MMA covers 32 bytes
// of K (K = 32 for kind::f8f6f4, 8 for kind::tf32), so every shared-memory
// offset is the same and only the element count of a k-block changes.
enum { KIND_F16 = 0, KIND_F8 = 1, KIND_TF32 = 2 };
template <int KIND> struct KBlock { static constexpr int elems = KIND == KIND_F8 ? 128 : KIND == KIND_TF32 ? 32 : 64; };

// One MMA of the operand kind, issued by the CTA (PAIR false) or by the
// leader of a CTA pair (PAIR true).
template <int KIND, bool PAIR>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc)
{
    if constexpr (PAIR) {
        if constexpr (KIND == KIND_F8) ptx::mma_f8_ss_pair(d_tmem, ad, bd, idesc, acc);
        else if constexpr (KIND == KIND_TF32) ptx::mma_tf32_ss_pair(d_tmem, ad, bd, idesc, acc);
        else ptx::mma_f16_ss_pair(d_tmem, ad, bd, idesc, acc);
    } else {
        if constexpr (KIND == KIND_F8) ptx::mma_f8_ss(d_tmem, ad, bd, idesc, acc);
        else if constexpr (KIND == KIND_TF32) ptx::mma_tf32_ss(d_tmem, ad, bd, idesc, acc);
        else ptx::mma_f16_ss(d_tmem, ad, bd, idesc, acc);
    }
}
constexpr int kThreads = 192;      // 6 warps
constexpr int kEpiWarps = 4;
constexpr uint32_t kStageCBytes = 32 * 128;   // one staged 32-row x 128-byte block of C

// ---- shared-memory matrix descriptors (tcgen05, 128-byte swizzle) -----------
//
// Bits 0-13 start address >> 4, 16-29 leading-dimension byte offset >> 4,
// 32-45 stride-dimension byte offset >> 4, 46-47 version (1), 49-51 base
// offset (0: every swizzle atom starts 1024-byte aligned), 61-63 layout
// (2 = 128-byte swizzle).
__host__ __device__ constexpr uint64_t desc_sw128(uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    return ((uint64_t)((lbo_bytes >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo_bytes >> 4) & 0x3fffu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ uint64_t desc_at(uint64_t tmpl, uint32_t smem_byte_addr)
{
    return tmpl | (uint64_t)((smem_byte_addr >> 4) & 0x3fffu);
}

// K-major operand (rows of 64 K-elements = 128 bytes, 8-row swizzle atoms
// 1024 bytes apart).  The leading offset is unused for swizzled K-major
// layouts; the usual value 16 bytes is kept.
constexpr uint64_t kDescKMajor = desc_sw128(16, 1024);
// MN-major operand (B stored K x N): each 64-wide column block is 64 k-rows
// of 128 bytes (8 KiB); the leading offset steps between 64-wide column
// blocks, the stride offset between 8-row K groups.
constexpr uint64_t kDescMNMajor = desc_sw128(kBK * 128, 1024);

// ---- instruction descriptor (kind::f16) -------------------------------------
//
// Bits 4-5 D type (1 = F32), 7-9 A type and 10-12 B type (kind::f16: 0 F16,
// 1 BF16; kind::f8f6f4: 0 E4M3, 1 E5M2; kind::tf32: 2 TF32), 15 A major and
// 16 B major (0 = K, 1 = MN), 17-22 N >> 3, 24-28 M >> 4.  The same layout
// serves the three kinds.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_type, bool b_mn_major, int m, int n,
                                                  bool a_mn_major = false)
{
    return (1u << 4) | ((ab_type & 7u) << 7) | ((ab_type & 7u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

// ---- shared-memory plan ---------------------------------------------------
template <int BN, int STAGES>
struct SmemPlan {
    static constexpr uint32_t a_stage = kBM * kBK * 2;
    static constexpr uint32_t b_stage = BN * kBK * 2;
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = a_off + STAGES * a_stage;
    static constexpr uint32_t c_off = b_off + STAGES * b_stage;
    static constexpr uint32_t bar_off = c_off + kEpiWarps * 2 * kStageCBytes;
    // full[S], empty[S], tmem_full[2], tmem_empty[2], drain, C_in loads[4 epilogue warps]
    static constexpr uint32_t n_bars = 2 * STAGES + 5 + kEpiWarps;
    static constexpr uint32_t slot_off = bar_off + 8 * n_bars;   // TMEM address
    static constexpr uint32_t abort_off = slot_off + 4;
    static constexpr uint32_t flag_off = abort_off + 4;          // epilogue broadcast word
    static constexpr uint32_t bytes = flag_off + 4;
    static constexpr uint32_t alloc_bytes = bytes + 1024;        // slack to align the base to 1024
};

// SM-clock record for benchmarks (tgemm_debug_clock_record): CTA 0's
// thread 0 notes %globaltimer and %clock64 once its dependency wait returns
// and, as the CTA leaves, adds the elapsed nanoseconds and SM cycles (and one
// launch) to rec[0..2].  Launches on a stream never overlap between those
// two points (the next launch's wait returns only once this one is
// complete), so the sums give the average SM clock over the launches that
// ran while the record was set.  One uniform branch when it is not set.
__device__ __forceinline__ void clock_record_begin(const GemmParams &p)
{
    if (p.clock_rec != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        p.clock_rec[4] = ptx::globaltimer_ns();
        p.clock_rec[5] = clock64();
    }
}

__device__ __forceinline__ void clock_record_end(const GemmParams &p)
{
    if (p.clock_rec != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
        const uint64_t t1 = ptx::globaltimer_ns();
        const uint64_t c1 = clock64();
        atomicAdd(reinterpret_cast<unsigned long long *>(&p.clock_rec[0]),
                  (unsigned long long)(t1 - p.clock_rec[4]));
        atomicAdd(reinterpret_cast<unsigned long long *>(&p.clock_rec[1]),
                  (unsigned long long)(c1 - p.clock_rec[5]));
        atomicAdd(reinterpret_cast<unsigned long long *>(&p.clock_rec[2]), 1ull);
    }
}

template <int BN>
struct TmemCols {
    static constexpr uint32_t value = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                      : (2 * BN <= 256) ? 256 : 512;
};

__device__ __forceinline__ uint32_t pack_out(float lo, float hi, int out)
{
    uint32_t u;
    if (out == OUT_F16) {
        __half2 h = __floats2half2_rn(lo, hi);
        memcpy(&u, &h, 4);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        memcpy(&u, &h, 4);
    }
    return u;
}

// ---- fused epilogue ----------------------------------------------------------
//
// D = act(alpha * acc + beta * C_in + bias[col]) in FP32 before the cast: the
// epilogue fusion the Croqtile tutorial credits cuBLAS with (its comparison
// with cuBLAS), in the usual affine-plus-activation form.  GELU uses its tanh
// form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
// Unpack two 16-bit output-type values (low, high) to floats.
__device__ __forceinline__ float2 unpack_out(uint32_t u, int out)
{
    if (out == OUT_F16) {
        __half2 h;
        memcpy(&h, &u, 4);
        return __half22float2(h);
    }
    __nv_bfloat162 h;
    memcpy(&h, &u, 4);
    return __bfloat1622float2(h);
}

__device__ __forceinline__ float load_bias(const void *b, int dt, int64_t j)
{
    if (dt == OUT_F32) return __ldg(static_cast<const float *>(b) + j);
    if (dt == OUT_F16) return __half2float(__ldg(static_cast<const __half *>(b) + j));
    return __bfloat162float(__ldg(static_cast<const __nv_bfloat16 *>(b) + j));
}

// GELU's tanh form rewritten with 0.5 (1 + tanh(u)) = 1 / (1 + exp(-2u)):
// x / (1 + exp(-2u)), u = sqrt(2/pi) (x + 0.044715 x^3).  exp overflows to
// +inf for very negative x, which gives the limit 0.
__device__ __forceinline__ float act_apply(float x, int act)
{
    if (act == 1) return fmaxf(x, 0.f);
    if (act == 2) {
        const float u = 0.7978845608f * fmaf(0.044715f * x * x, x, x);
        return __fdividef(x, 1.f + __expf(-2.f * u));
    }
    return x;
}

// The epilogue's scalars in registers.  Loops that interleave shared-memory
// stores (asm with a memory clobber) with reads of the launch parameters made
// the compiler re-read the parameters per element; the per-chunk loops take
// this copy instead.  Member names match GemmParams, so the helpers below
// accept either.
struct EpiScalars {
    const void *bias;
    int32_t N;
    int32_t bias_dtype;
    float alpha, beta;
    int32_t act;
    int32_t epi;
    __device__ __forceinline__ static EpiScalars of(const GemmParams &p)
    {
        return EpiScalars{p.bias, p.N, p.bias_dtype, p.alpha, p.beta, p.act, p.epi};
    }
};

template <class P>
__device__ __forceinline__ float epi_combine(const P &p, float acc, float cin, float bias)
{
    float r = p.alpha * acc;
    if (p.epi & 2) r = fmaf(p.beta, cin, r);
    return act_apply(r + bias, p.act);
}

template <class P>
__device__ __forceinline__ float epi_value(const P &p, float acc, float cin, int64_t col)
{
    const float b = (p.bias && col < p.N) ? load_bias(p.bias, p.bias_dtype, col) : 0.f;
    return epi_combine(p, acc, cin, b);
}

// Bias values of columns [col, col + n) (n = 4 or 8), zero past N or without
// a bias; one or two 16-byte loads when the run lies inside the vector.
template <int n, class P>
__device__ __forceinline__ void load_bias_run(const P &p, int64_t col, float (&out)[n])
{
    if (!p.bias) {
#pragma unroll
        for (int t = 0; t < n; ++t) out[t] = 0.f;
        return;
    }
    if (col + n <= p.N) {
        if (p.bias_dtype == OUT_F32) {
            const float4 *b = reinterpret_cast<const float4 *>(static_cast<const float *>(p.bias) + col);
#pragma unroll
            for (int h = 0; h < n / 4; ++h) {
                const float4 v = __ldg(b + h);
                out[4 * h] = v.x, out[4 * h + 1] = v.y, out[4 * h + 2] = v.z, out[4 * h + 3] = v.w;
            }
        } else if constexpr (n == 8) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.bias) + col));
            const float2 a = unpack_out(v.x, p.bias_dtype), b = unpack_out(v.y, p.bias_dtype);
            const float2 c = unpack_out(v.z, p.bias_dtype), d = unpack_out(v.w, p.bias_dtype);
            out[0] = a.x, out[1] = a.y, out[2] = b.x, out[3] = b.y, out[4] = c.x, out[5] = c.y, out[6] = d.x, out[7] = d.y;
        } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(p.bias) + col));
            const float2 a = unpack_out(v.x, p.bias_dtype), b = unpack_out(v.y, p.bias_dtype);
            out[0] = a.x, out[1] = a.y, out[2] = b.x, out[3] = b.y;
        }
        return;
    }
#pragma unroll
    for (int t = 0; t < n; ++t) out[t] = col + t < p.N ? load_bias(p.bias, p.bias_dtype, col + t) : 0.f;
}

__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// Per-warp state for reading C_in through the staging block.
struct EpiCtx {
    const GemmParams *p;    // null: write the raw FP32 values (stream-K partials)
    uint32_t cin_bar;       // this warp's mbarrier for C_in loads
    uint32_t cin_phase;     // loads issued so far (parity)
    WaitCtx wc;
    int32_t z = 0;          // batch coordinate of the current tile
};

// Tile number -> (batch, tile row, tile column): batches are consecutive runs
// of tiles_per_batch tile numbers, each walked in grouped order.
__device__ __forceinline__ void batched_tile(const GemmParams &p, int tile, int &b, int64_t &tr, int64_t &tc)
{
    b = tile / p.tiles_per_batch;
    int32_t r, c;
    grouped_tile32(p.tiles_m, p.tiles_n, p.group_m, tile - b * p.tiles_per_batch, r, c);
    tr = r;
    tc = c;
}

// Fetch the C_in block (x, row0) of this warp into the staging block `sbuf`
// and wait for it.  Returns false if the wait timed out.
__device__ __forceinline__ bool fetch_cin(EpiCtx &e, uint32_t sbuf, int32_t x, int32_t row0, int lane)
{
    if (lane == 0) {
        ptx::mbar_arrive_expect_tx(e.cin_bar, kStageCBytes);
        ptx::tma_load_3d(sbuf, &e.p->tma_cin, e.cin_bar, x, row0, e.z);
    }
    const bool ok = wait_bounded(e.cin_bar, e.cin_phase & 1u, e.wc, SITE_EPI_CIN);
    ++e.cin_phase;
    return __all_sync(0xffffffffu, ok);
}

// Cast one 128-byte-wide column chunk of this warp's 32 rows (v0, plus v1
// for 16-bit output: 64 columns), stage it in one of the warp's two swizzled
// staging blocks and store it with TMA at (x, row0) of `map`; rows >= rows_lim
// or a chunk starting at x >= cols_lim are not written (TMA clips the rest).
// `cc` counts chunks and selects the staging block.
template <int OUT>
__device__ __forceinline__ void stage_store_chunk(const CUtensorMap *map, int32_t rows_lim, int32_t cols_lim,
                                                  uint32_t stage_base, uint32_t &cc, int32_t row0, int32_t x,
                                                  int lane, uint32_t (&v0)[32], uint32_t (&v1)[32], EpiCtx &e)
{
    const uint32_t sbuf = stage_base + (cc & 1u) * kStageCBytes;
    if (lane == 0) ptx::bulk_wait_group_read<1>();   // the store that last used sbuf is done reading
    __syncwarp();
    const uint32_t row_addr = sbuf + lane * 128;
    const bool fused = e.p != nullptr && (e.p->epi & 1);
    const bool with_cin = fused && (e.p->epi & 2) && fetch_cin(e, sbuf, x, row0, lane);
    const EpiScalars es = fused ? EpiScalars::of(*e.p) : EpiScalars{};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t addr = row_addr + ((uint32_t)(j ^ (lane & 7)) << 4);   // 128-byte swizzle
        uint32_t w0, w1, w2, w3;
        if constexpr (OUT == OUT_F32) {
            if (fused) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                if (with_cin) {
                    const uint4 q = ld_shared_u4(addr);
                    c[0] = __uint_as_float(q.x), c[1] = __uint_as_float(q.y);
                    c[2] = __uint_as_float(q.z), c[3] = __uint_as_float(q.w);
                }
                float bv[4];
                load_bias_run<4>(es, (int64_t)x + 4 * j, bv);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    v0[4 * j + t] = __float_as_uint(epi_combine(es, __uint_as_float(v0[4 * j + t]), c[t], bv[t]));
            }
            w0 = v0[4 * j + 0];
            w1 = v0[4 * j + 1];
            w2 = v0[4 * j + 2];
            w3 = v0[4 * j + 3];
        } else {
            // columns 8j .. 8j+7 of the 64-column chunk
            uint32_t *src = j < 4 ? &v0[8 * j] : &v1[8 * (j - 4)];
            if (fused) {
                float c[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (with_cin) {
                    const uint4 q = ld_shared_u4(addr);
                    const float2 c0 = unpack_out(q.x, OUT), c1 = unpack_out(q.y, OUT);
                    const float2 c2 = unpack_out(q.z, OUT), c3 = unpack_out(q.w, OUT);
                    c[0] = c0.x, c[1] = c0.y, c[2] = c1.x, c[3] = c1.y, c[4] = c2.x, c[5] = c2.y, c[6] = c3.x, c[7] = c3.y;
                }
                float bv[8];
                load_bias_run<8>(es, (int64_t)x + 8 * j, bv);
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    src[t] = __float_as_uint(epi_combine(es, __uint_as_float(src[t]), c[t], bv[t]));
            }
            w0 = pack_out(__uint_as_float(src[0]), __uint_as_float(src[1]), OUT);
            w1 = pack_out(__uint_as_float(src[2]), __uint_as_float(src[3]), OUT);
            w2 = pack_out(__uint_as_float(src[4]), __uint_as_float(src[5]), OUT);
            w3 = pack_out(__uint_as_float(src[6]), __uint_as_float(src[7]), OUT);
        }
        ptx::st_shared_v4(addr, w0, w1, w2, w3);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (x < cols_lim && row0 < rows_lim) ptx::tma_store_3d(map, sbuf, x, row0, e.z);
        ptx::bulk_commit_group();
    }
    ++cc;
}

// Drain one accumulator buffer held in this warp's TMEM lane quarter: tile
// rows [row0, row0 + 32), columns [col0, col0 + BN), into `map` (C, or the
// FP32 partial-tile workspace).  Each 128-byte-wide column chunk is read with
// tcgen05.ld and handed to stage_store_chunk.  `release()` runs on lane 0
// once the last chunk is in registers, handing the buffer back to the MMA
// issuer.
template <int BN, int OUT, typename Release>
__device__ __forceinline__ void epilogue_drain(const CUtensorMap *map, int32_t rows_lim, int32_t cols_lim,
                                               uint32_t t_acc, uint32_t stage_base, uint32_t &cc, int32_t row0,
                                               int32_t col0, int lane, Release release, EpiCtx &e)
{
    constexpr int kOutBytes = OUT == OUT_F32 ? 4 : 2;
    constexpr int kChunkCols = 128 / kOutBytes;          // columns of one 128-byte staged row
    constexpr int kChunks = BN / kChunkCols;
#pragma unroll 1
    for (int c = 0; c < kChunks; ++c) {
        uint32_t v0[32], v1[32];
        ptx::tmem_ld_32x32b_x32(t_acc + c * kChunkCols, v0);
        if constexpr (kChunkCols == 64) ptx::tmem_ld_32x32b_x32(t_acc + c * kChunkCols + 32, v1);
        ptx::tmem_ld_wait();
        if (c == kChunks - 1) {
            // The accumulator buffer is fully read: hand it back.
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) release();
        }
        stage_store_chunk<OUT>(map, rows_lim, cols_lim, stage_base, cc, row0, col0 + c * kChunkCols, lane, v0, v1, e);
    }
}

// CTAs of the one-CTA tile kernel resident per SM: two for the two-stage
// 128 x 128 ring (98 KB of shared memory and 256 TMEM columns each), one
// otherwise.  Tiles with one or two k-blocks (K <= 128) spend most of their
// time in the epilogue; a second CTA doubles the epilogue warps per SM.
template <int BN, int STAGES>
struct TileResidency {
    static constexpr int ctas_per_sm = (BN == 128 && STAGES <= 2) ? 2 : 1;
};

template <int BN, int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
__global__ void __launch_bounds__(kThreads, TileResidency<BN, STAGES>::ctas_per_sm)
    gemm_persistent_kernel(const __grid_constant__ GemmParams p)
{
    static_assert(KIND == KIND_F16 || !B_MN, "FP8 and TF32 operands are K-major only");
    using Plan = SmemPlan<BN, STAGES>;
    constexpr uint32_t kStageBytes = Plan::a_stage + Plan::b_stage;
    constexpr uint32_t kTmemCols = TmemCols<BN>::value;
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64, 128, 192 or 256");
    static_assert(2 * BN <= 512, "two accumulator buffers must fit in tensor memory");
    static_assert(Plan::alloc_bytes <= 232448, "shared memory plan exceeds 227 KiB");
    static_assert(TileResidency<BN, STAGES>::ctas_per_sm == 1 ||
                      (Plan::alloc_bytes <= 232448 / 2 - 1024 && 2 * kTmemCols <= 512),
                  "two CTAs of this plan must fit one SM");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base + Plan::a_off;
    const uint32_t sB = base + Plan::b_off;
    const uint32_t sC = base + Plan::c_off;
    const uint32_t bar = base + Plan::bar_off;
    auto full_bar = [&](int s) { return bar + 8u * s; };
    auto empty_bar = [&](int s) { return bar + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar + 8u * (2 * STAGES + 4);
    const uint32_t slot = base + Plan::slot_off;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_ptr + Plan::abort_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), kEpiWarps);
        }
        ptx::mbar_init(drain_bar, 1);
        for (int w = 0; w < kEpiWarps; ++w) ptx::mbar_init(drain_bar + 8u * (1 + w), 1);   // C_in loads
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&p.tma_a);
        ptx::prefetch_tensormap(&p.tma_b);
        ptx::prefetch_tensormap(&p.tma_c);
    }
    if (warp == 1) {
        ptx::tmem_alloc(slot, kTmemCols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before_sync();
    }
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(base_ptr + Plan::slot_off);

    const WaitCtx wc{p.status, abort_flag, p.timeout_ns};
    const int num_tiles = p.num_tiles;
    ptx::grid_dependency_wait();   // inputs written and outputs read by earlier kernels are settled
    clock_record_begin(p);
    ptx::launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, issued_parity = 0;   // latest load per stage, for wind-down
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int64_t tr, tc;
                int bz;
                batched_tile(p, tile, bz, tr, tc);
                const int32_t m0 = (int32_t)tr * kBM;
                const int32_t n0 = (int32_t)tc * BN;
                const int32_t za = p.a_batched ? bz : 0, zb = p.b_batched ? bz : 0;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, wc, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(s);
                    ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                    const int32_t k0 = kb * KBlock<KIND>::elems;
                    ptx::tma_load_3d(sA + s * Plan::a_stage, &p.tma_a, fb, k0, m0, za);
                    if (B_MN) {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            ptx::tma_load_3d(sB + s * Plan::b_stage + j * (kBK * 128), &p.tma_b, fb,
                                             n0 + 64 * j, k0, zb);
                    } else {
                        ptx::tma_load_3d(sB + s * Plan::b_stage, &p.tma_b, fb, k0, n0, zb);
                    }
                    issued_mask |= 1u << s;
                    issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Wind down: wait for the copies still in flight into our ring.
                for (int t = 0; t < STAGES; ++t)
                    if (issued_mask & (1u << t))
                        wait_bounded(full_bar(t), (issued_parity >> t) & 1u, wc, SITE_DRAIN_LOADS, false);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t local = 0;      // tiles done by this CTA
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
                const uint32_t buf = local & 1u;
                const uint32_t bph = (local >> 1) & 1u;
                if (!wait_bounded(tempty_bar(buf), bph ^ 1u, wc, SITE_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < p.num_kb;) {
                    // Two k-blocks in adjacent stages per pass when the second
                    // one's data is already in (one fence, one loop overhead for
                    // both): the lone issuing thread's per-k-block overhead would
                    // otherwise idle the tensor pipe.  The second stage is only
                    // tested, never waited for, so a tile's first MMAs are not
                    // held back while the ring fills.
                    if (!wait_bounded(full_bar(s), ph, wc, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    const int n =
                        (kb + 1 < p.num_kb && s + 1 < STAGES && ptx::mbar_test_wait(full_bar(s + 1), ph)) ? 2 : 1;
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < n) {
                            const uint32_t a_addr = sA + (s + h) * Plan::a_stage;
                            const uint32_t b_addr = sB + (s + h) * Plan::b_stage;
#pragma unroll
                            for (int k = 0; k < kBK / kUmmaK; ++k) {
                                const uint64_t ad = desc_at(kDescKMajor, a_addr + k * (kUmmaK * 2));
                                const uint64_t bd = B_MN ? desc_at(kDescMNMajor, b_addr + k * (kUmmaK * 128))
                                                         : desc_at(kDescKMajor, b_addr + k * (kUmmaK * 2));
                                mma_issue<KIND, false>(d_tmem, ad, bd, p.idesc, ((kb + h) | k) != 0 ? 1u : 0u);
                            }
                            ptx::mma_commit(empty_bar(s + h));   // stage reusable once these MMAs finish
                        }
                    }
                    kb += n;
                    s += n;
                    if (s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(tfull_bar(buf));         // accumulator ready for the epilogue
            }
            if (!ok) {
                // Wind down: every MMA issued so far must finish before the
                // tensor memory is released.
                ptx::mma_commit(drain_bar);
                wait_bounded(drain_bar, 0, wc, SITE_DRAIN_MMA, false);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;                         // staging slot 0..3
        const int q = warp & 3;                          // TMEM lane quarter = tile rows 32q..32q+31
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t stage_base = sC + ew * 2 * kStageCBytes;
        EpiCtx ectx{&p, drain_bar + 8u * (1 + ew), 0u, wc};
        uint32_t local = 0, cc = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const uint32_t buf = local & 1u;
            const uint32_t bph = (local >> 1) & 1u;
            const bool got = wait_bounded(tfull_bar(buf), bph, wc, SITE_EPI_TMEM_FULL);
            if (!__all_sync(0xffffffffu, got)) break;
            ptx::tc_fence_after_sync();

            int64_t tr, tc;
            int bz;
            batched_tile(p, tile, bz, tr, tc);
            ectx.z = bz;
            const int32_t row0 = (int32_t)tr * kBM + 32 * q;
            const int32_t col0 = (int32_t)tc * BN;
            const uint32_t t_acc = tmem_base + lane_base + buf * BN;
            const uint32_t release_bar = tempty_bar(buf);
            epilogue_drain<BN, OUT>(&p.tma_c, p.M, p.N, t_acc, stage_base, cc, row0, col0, lane,
                                    [&] { ptx::mbar_arrive(release_bar); }, ectx);
        }
        if (lane == 0) ptx::bulk_wait_group_all();
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
    clock_record_end(p);
}

template <int BN, int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
cudaError_t launch_gemm(const GemmParams &p, int grid, cudaStream_t stream)
{
    auto kern = gemm_persistent_kernel<BN, STAGES, OUT, B_MN, KIND>;
    constexpr uint32_t smem = SmemPlan<BN, STAGES>::alloc_bytes;
    static std::atomic<unsigned long long> smem_set{0};
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see ptx::grid_dependency_wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// max_active stays null: the one-CTA grid is sized from the SM count and
// TileResidency (run_body).
#define TGEMM_VARIANT(BN, ST, OUT, BMN) \
    {BN, ST, OUT, BMN, SmemPlan<BN, ST>::alloc_bytes, &launch_gemm<BN, ST, OUT, (BMN) != 0>, 1, nullptr}
#define TGEMM_VARIANT_KIND(BN, ST, OUT, KIND) \
    {BN, ST, OUT, 0, SmemPlan<BN, ST>::alloc_bytes, &launch_gemm<BN, ST, OUT, false, KIND>, 1, nullptr, KIND}

}  // namespace tgemm
