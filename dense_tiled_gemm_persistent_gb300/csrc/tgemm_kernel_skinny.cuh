// Skinny GEMM (a handful of rows of A, e.g. 16 tokens through a projection):
// swap-AB plus split-K.
//
// With M = 16 a 128-row tile would leave 7/8 of every MMA empty and only
// N/BN CTAs would stream the weights.  Instead the kernel computes
// C^T = B^T * A^T: the weight rows (N) feed the MMA's M = 128 side and the
// M tokens, padded to NPAD (16, 32 or 64), become the MMA's N.  K is cut into
// `splits` runs of whole 64-deep k-blocks so that tiles_n * splits CTAs (two
// to three per SM) stream the weight matrix from HBM at once.  This is a
// memory-bound shape: about 16 FLOP per byte, far under the tensor ridge
// (the roofline argument of the wmrh.cn essay on GEMM tiling, sections 1.1
// and 3.3); splitting K is this library's own choice, not from the pages.
//
// Every CTA accumulates its partial D (128 weight rows x NPAD tokens, FP32)
// in tensor memory.  With one split it casts and stores C directly.
// Otherwise it writes the partial to a workspace, fences, and bumps the
// tile's arrival counter; the CTA that arrives last sums the `splits`
// partials in split order 0, 1, ..., splits-1 (a fixed order, so results do
// not depend on which CTA finishes last), casts with round-to-nearest-even,
// writes C and resets the counter to zero for the next call.  Nobody waits
// for another CTA.
#pragma once

#include "tgemm_kernel.cuh"

namespace tgemm {

constexpr int kSkinnyStages = 4;
constexpr int kSkinnyRows = 128;      // weight rows (C columns) per CTA

template <int NPAD>
struct SkinnyPlan {
    static constexpr uint32_t w_stage = kSkinnyRows * kBK * 2;   // 16 KiB
    static constexpr uint32_t x_stage = NPAD * kBK * 2;          // 2, 4 or 8 KiB
    static constexpr uint32_t w_off = 0;
    static constexpr uint32_t x_off = w_off + kSkinnyStages * w_stage;
    static constexpr uint32_t bar_off = x_off + kSkinnyStages * x_stage;
    static constexpr uint32_t n_bars = 2 * kSkinnyStages + 3;     // full, empty, tmem_full, drain x 2
    static constexpr uint32_t slot_off = bar_off + 8 * n_bars;
    static constexpr uint32_t abort_off = slot_off + 4;
    static constexpr uint32_t last_off = abort_off + 4;
    static constexpr uint32_t fail_off = last_off + 4;
    static constexpr uint32_t bytes = fail_off + 4;
    static constexpr uint32_t alloc_bytes = bytes + 1024;
};

// L2 prefetch of the first `depth` k-blocks of this CTA's weight slice,
// issued by the producer before griddepcontrol.wait.  A CTA of a dependent
// launch is resident while the previous kernel still runs (the half-size ring
// leaves room for two CTAs per SM), so its weights stream from HBM during the
// previous kernel's tail instead of after it.  Weights are read-only inputs
// of the product; even if an earlier kernel were still writing them, the
// prefetch only warms L2 and the TMA loads after the wait read the current
// data.  How deep to prefetch depends on when the dependent launch starts
// (GemmParams::late_trigger): started at once, only the first
// kSkinnyPrefetchKb k-blocks, since a whole slice would compete with the
// running launch for all of its time (measured over the M <= 64 picker grid,
// best configuration per point, geometric mean: no prefetch +3.6 %, 2
// k-blocks +1.0 %, 8 +1.6 %, whole slices +2.4 % against 4); started once
// the running launch has issued its last loads, the whole slice.
constexpr int kSkinnyPrefetchKb = 4;

// MMA issue of the swap-AB kernels.  With 128 weight rows x NPAD tokens per
// instruction the tensor pipe finishes an MMA in about 40 SM cycles, and a
// single issuing thread cannot keep up: measured on a GB300, one thread
// spends about 45 cycles per tcgen05.mma with operands that are constant
// offsets, about 64 when they come from a runtime stage index, and per
// k-block another ~140 waiting on an already completed full barrier and ~45
// committing to the empty one -- 450 to 550 cycles per 16 KiB k-block in
// all, which bounded the kernel (a run with the loads taken out was as slow
// as the whole kernel).  So two threads issue: warp 1 and warp 2 (lane 0),
// the ring stages of even and odd index, each waiting for and committing
// only its own stages (a stage is always served by the same thread, so its
// full barrier's phases are waited on in order), the ring loop unrolled so
// that stage offsets are constants.  Two issuers measured 57 cycles per MMA
// against 93 for one with the same waits and commits.
constexpr int kSkinnyIssuers = 2;

// Each issuer adds into its own accumulators (NPAD TMEM columns apart): two
// for NPAD <= 32 (k-step j into accumulator j mod 2), one for 64 and 128.
// The epilogue adds them in a fixed order (0, 1, ...), so results do not
// depend on timing.  Column budgets (64, 128, 128, 256 for NPAD 16, 32, 64,
// 128) keep four CTAs per SM (two at NPAD 128) within 512 TMEM columns.
template <int NPAD>
struct SkinnyAcc {
    static constexpr int per_issuer = NPAD <= 32 ? 2 : 1;
    static constexpr int count = kSkinnyIssuers * per_issuer;
    static constexpr uint32_t tmem_cols = count * NPAD < 32 ? 32u : (uint32_t)(count * NPAD);
    static_assert((kBK / kUmmaK) % per_issuer == 0, "every k-block writes each of its issuer's accumulators");
};

// The MMA role of issuer `me` (0 or 1) over k-blocks kb0..kb1: full
// barriers at bar + 8 s, empty ones at bar + 8 (S + s) for ring stage s; W
// and X stages W_STAGE and X_STAGE bytes apart from sW and sX.  Ends with a
// commit to tfull_bar (initialised for kSkinnyIssuers arrivals), or -- when
// a wait ran out -- to the issuer's own drain barrier, waited on before
// returning so that no MMA of this thread is still reading the ring.
// Returns whether every wait completed.
template <int NPAD, bool W_MN, int S, uint32_t W_STAGE, uint32_t X_STAGE, int KIND = KIND_F16>
__device__ __forceinline__ bool skinny_mma_role(int me, uint32_t sW, uint32_t sX, uint32_t bar, uint32_t tfull_bar,
                                                uint32_t drain_bar, int kb0, int kb1, uint32_t tmem_base,
                                                uint32_t idesc, const WaitCtx &wc)
{
    constexpr int P = SkinnyAcc<NPAD>::per_issuer;
    static_assert(S >= 2, "both issuers own a stage");
    const uint32_t d0 = tmem_base + (uint32_t)(me * P * NPAD);
    bool ok = true, fresh = true;
    uint32_t ph = 0;
    for (int kr = kb0; ok && kr < kb1; kr += S, ph ^= 1u) {   // one pass over the ring
#pragma unroll
        for (int s = 0; s < S; ++s) {
            if (kr + s >= kb1) break;
            if ((s & 1) != me) continue;
            if (!wait_bounded(bar + 8u * s, ph, wc, SITE_MMA_FULL)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            const uint32_t w_addr = sW + s * W_STAGE;
            const uint32_t x_addr = sX + s * X_STAGE;
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
                const uint64_t ad = W_MN ? desc_at(kDescMNMajor, w_addr + k * (kUmmaK * 128))
                                         : desc_at(kDescKMajor, w_addr + k * (kUmmaK * 2));
                const uint64_t bd = desc_at(kDescKMajor, x_addr + k * (kUmmaK * 2));
                // the issuer's first k-block overwrites each of its accumulators
                const uint32_t acc = (fresh && k < P) ? 0u : 1u;
                if constexpr (KIND == KIND_F8) ptx::mma_f8_ss(d0 + (uint32_t)((k % P) * NPAD), ad, bd, idesc, acc);
                else ptx::mma_f16_ss(d0 + (uint32_t)((k % P) * NPAD), ad, bd, idesc, acc);
            }
            ptx::mma_commit(bar + 8u * (S + s));
            fresh = false;
        }
    }
    if (ok) {
        ptx::mma_commit(tfull_bar);
    } else {
        ptx::mma_commit(drain_bar);
        wait_bounded(drain_bar, 0, wc, SITE_DRAIN_MMA, false);
    }
    return ok;
}

// This warp's 32 TMEM lanes (taddr carries the lane offset) of the summed
// accumulators into v[0..NPAD).  A K range of one k-block (ring stage 0
// only) leaves the second issuer's accumulators unwritten: only the first
// issuer's are read then.
template <int NPAD>
__device__ __forceinline__ void load_skinny_acc(uint32_t taddr, int kblocks, float (&v)[NPAD])
{
    constexpr int A = SkinnyAcc<NPAD>::count;
    constexpr int P = SkinnyAcc<NPAD>::per_issuer;
    const bool second = kblocks >= 2;
#pragma unroll
    for (int c = 0; c < NPAD / 16; ++c) {
        uint32_t r[A][16];
#pragma unroll
        for (int a = 0; a < A; ++a)
            if (a < P || second) ptx::tmem_ld_32x32b_x16(taddr + a * NPAD + 16 * c, r[a]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float t = __uint_as_float(r[0][j]);
#pragma unroll
            for (int a = 1; a < A; ++a)
                if (a < P || second) t += __uint_as_float(r[a][j]);
            v[16 * c + j] = t;
        }
    }
}

template <bool W_MN, int KE = kBK>
__device__ __forceinline__ void prefetch_weights_l2(const CUtensorMap *tma_b, int32_t n0, int kb0, int kb1,
                                                    int depth)
{
    const int kbe = kb1 - kb0 > depth ? kb0 + depth : kb1;
    for (int kb = kb0; kb < kbe; ++kb) {
        const int32_t k0 = kb * KE;   // KE elements per 128-byte k-block row
        if (W_MN) {
#pragma unroll
            for (int j = 0; j < kSkinnyRows / 64; ++j) ptx::tma_prefetch_l2_2d(tma_b, n0 + 64 * j, k0);
        } else {
            ptx::tma_prefetch_l2_2d(tma_b, k0, n0);
        }
    }
}

template <int OUT>
__device__ __forceinline__ void store_out(void *c, int64_t idx, float v)
{
    if constexpr (OUT == OUT_F32) {
        static_cast<float *>(c)[idx] = v;
    } else if constexpr (OUT == OUT_F16) {
        static_cast<__half *>(c)[idx] = __float2half_rn(v);
    } else {
        static_cast<__nv_bfloat16 *>(c)[idx] = __float2bfloat16_rn(v);
    }
}

// One output element into shared memory (shared-window address), rounded
// to nearest even for 16-bit outputs.
template <int OUT>
__device__ __forceinline__ void st_shared_out(uint32_t addr, float v)
{
    if constexpr (OUT == OUT_F32) {
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
    } else {
        unsigned short h;
        if constexpr (OUT == OUT_F16) h = __half_as_ushort(__float2half_rn(v));
        else h = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(h) : "memory");
    }
}

// C[m][n] = v with the fused epilogue (when enabled): C_in read with a
// plain load, bias by output column n.
template <int OUT>
__device__ __forceinline__ float epi_apply(const GemmParams &p, int m, int64_t n, float v)
{
    if (p.epi & 1) {
        float cin = 0.f;
        if (p.epi & 2) {
            const int64_t ci = (int64_t)m * p.ldc_in + n;
            if constexpr (OUT == OUT_F32) cin = static_cast<const float *>(p.cin_ptr)[ci];
            else if constexpr (OUT == OUT_F16) cin = __half2float(static_cast<const __half *>(p.cin_ptr)[ci]);
            else cin = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.cin_ptr)[ci]);
        }
        v = epi_value(p, v, cin, n);
    }
    return v;
}

template <int OUT>
__device__ __forceinline__ void store_out_epi(const GemmParams &p, int m, int64_t n, float v)
{
    store_out<OUT>(p.c_ptr, (int64_t)m * p.ldc + n, epi_apply<OUT>(p, m, n, v));
}

// Rows 0 .. rows-1 of column n of C from registers: the fused epilogue
// first, then the stores, with the pointer and pitch held in registers.
// (Interleaving stores with parameter reads made the compiler re-read the
// parameters per element: about 70 ns per row.)
template <int OUT, int NPAD>
__device__ __forceinline__ void store_column(const GemmParams &p, int rows, int64_t n, float (&v)[NPAD])
{
    if (p.epi & 1) {
#pragma unroll
        for (int m = 0; m < NPAD; ++m)
            if (m < rows) v[m] = epi_apply<OUT>(p, m, n, v[m]);
    }
    // a running row pointer: per-row offsets m * ldc held for all NPAD rows
    // at once spilled at NPAD 128
    constexpr int kOutBytes = OUT == OUT_F32 ? 4 : 2;
    char *row = static_cast<char *>(p.c_ptr) + n * kOutBytes;
    const int64_t pitch = p.ldc * kOutBytes;
#pragma unroll
    for (int m = 0; m < NPAD; ++m) {
        if (m < rows) store_out<OUT>(row, 0, v[m]);
        row += pitch;
    }
}

template <int NPAD, int OUT, bool W_MN>
__global__ void __launch_bounds__(kThreads) gemm_skinny_kernel(const __grid_constant__ GemmParams p)
{
    using Plan = SkinnyPlan<NPAD>;
    constexpr int S = kSkinnyStages;
    constexpr uint32_t kStageBytes = Plan::w_stage + Plan::x_stage;
    constexpr uint32_t kTmemCols = SkinnyAcc<NPAD>::tmem_cols;
    static_assert(NPAD == 16 || NPAD == 32 || NPAD == 64, "NPAD must be 16, 32 or 64");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sW = base + Plan::w_off;
    const uint32_t sX = base + Plan::x_off;
    const uint32_t bar = base + Plan::bar_off;
    auto full_bar = [&](int s) { return bar + 8u * s; };
    auto empty_bar = [&](int s) { return bar + 8u * (S + s); };
    const uint32_t tfull_bar = bar + 8u * (2 * S);
    const uint32_t drain_bar = bar + 8u * (2 * S + 1);    // first MMA issuer
    const uint32_t drain2_bar = bar + 8u * (2 * S + 2);   // second MMA issuer
    const uint32_t slot = base + Plan::slot_off;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_ptr + Plan::abort_off);
    volatile int *last_flag = reinterpret_cast<volatile int *>(base_ptr + Plan::last_off);
    volatile int *epi_fail = reinterpret_cast<volatile int *>(base_ptr + Plan::fail_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nt = blockIdx.x % p.tiles_n;
    const int split = blockIdx.x / p.tiles_n;
    const int kb0 = (int)((int64_t)split * p.num_kb / p.splits);
    const int kb1 = (int)((int64_t)(split + 1) * p.num_kb / p.splits);
    const int32_t n0 = nt * kSkinnyRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        ptx::mbar_init(tfull_bar, kSkinnyIssuers);
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(drain2_bar, 1);
        *abort_flag = 0;
        *last_flag = 0;
        *epi_fail = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&p.tma_a);
        ptx::prefetch_tensormap(&p.tma_b);
        prefetch_weights_l2<W_MN>(&p.tma_b, n0, kb0, kb1, kSkinnyPrefetchKb);
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
    ptx::grid_dependency_wait();   // inputs written and outputs read by earlier kernels are settled
    clock_record_begin(p);
    ptx::launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!wait_bounded(empty_bar(s), ph ^ 1u, wc, SITE_PRODUCER_EMPTY)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_bar(s);
                ptx::mbar_arrive_expect_tx(fb, kStageBytes);
                const int32_t k0 = kb * kBK;
                if (W_MN) {
#pragma unroll
                    for (int j = 0; j < kSkinnyRows / 64; ++j)
                        ptx::tma_load_2d(sW + s * Plan::w_stage + j * (kBK * 128), &p.tma_b, fb, n0 + 64 * j, k0);
                } else {
                    ptx::tma_load_2d(sW + s * Plan::w_stage, &p.tma_b, fb, k0, n0);
                }
                ptx::tma_load_2d(sX + s * Plan::x_stage, &p.tma_a, fb, k0, 0);
                issued_mask |= 1u << s;
                issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok)
                for (int t = 0; t < S; ++t)
                    if (issued_mask & (1u << t))
                        wait_bounded(full_bar(t), (issued_parity >> t) & 1u, wc, SITE_DRAIN_LOADS, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA, first issuer
        if (lane == 0)
            skinny_mma_role<NPAD, W_MN, S, Plan::w_stage, Plan::x_stage>(0, sW, sX, bar, tfull_bar, drain_bar, kb0,
                                                                         kb1, tmem_base, p.idesc, wc);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        if (warp == 2) {   // the second MMA issuer first
            if (lane == 0)
                skinny_mma_role<NPAD, W_MN, S, Plan::w_stage, Plan::x_stage>(1, sW, sX, bar, tfull_bar, drain2_bar,
                                                                             kb0, kb1, tmem_base, p.idesc, wc);
            __syncwarp();
        }
        const int q = warp & 3;                   // TMEM lanes 32q..32q+31 = weight rows
        const int nl = 32 * q + lane;             // row inside the 128-row tile
        const int64_t n = (int64_t)n0 + nl;
        const int M = p.M;
        const bool got = wait_bounded(tfull_bar, 0, wc, SITE_EPI_TMEM_FULL);
        if (!__all_sync(0xffffffffu, got) && lane == 0) *epi_fail = 1;
        ptx::named_barrier(1, 4 * 32);   // the four epilogue warps take one decision together
        if (!*epi_fail) {
            ptx::tc_fence_after_sync();
            float v[NPAD];
            load_skinny_acc<NPAD>(tmem_base + ((uint32_t)(32 * q) << 16), kb1 - kb0, v);
            if (p.splits == 1) {
                if (n < p.N) store_column<OUT, NPAD>(p, M, n, v);
            } else {
                // Partial of this split, [split][nt][row][NPAD]: each thread
                // owns one weight row and writes its NPAD sums contiguously.
                float4 *part = reinterpret_cast<float4 *>(
                    p.partials + (((int64_t)split * p.tiles_n + nt) * kSkinnyRows + nl) * NPAD);
#pragma unroll
                for (int c = 0; c < NPAD / 4; ++c)
                    part[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                __threadfence();
                ptx::named_barrier(1, 4 * 32);
                if (warp == 2 && lane == 0) {
                    const uint32_t prev = atomicAdd(&p.counters[nt], 1u);
                    *last_flag = prev == (uint32_t)(p.splits - 1) ? 1 : 0;
                }
                ptx::named_barrier(1, 4 * 32);
                if (*last_flag) {
                    __threadfence();
                    float acc[NPAD];
#pragma unroll
                    for (int m = 0; m < NPAD; ++m) acc[m] = 0.f;
                    const int64_t split_stride = (int64_t)p.tiles_n * kSkinnyRows * NPAD / 4;   // in float4
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.partials + ((int64_t)nt * kSkinnyRows + nl) * NPAD);
                    // Sum the partials in split order 0, 1, 2, ...; loads of up
                    // to four splits are issued before their additions.
                    int j = 0;
                    for (; j + 4 <= p.splits; j += 4) {
                        float4 t[4][NPAD / 4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int c = 0; c < NPAD / 4; ++c) t[u][c] = __ldcg(src + (j + u) * split_stride + c);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int c = 0; c < NPAD / 4; ++c) {
                                acc[4 * c] += t[u][c].x;
                                acc[4 * c + 1] += t[u][c].y;
                                acc[4 * c + 2] += t[u][c].z;
                                acc[4 * c + 3] += t[u][c].w;
                            }
                    }
                    for (; j < p.splits; ++j)
#pragma unroll
                        for (int c = 0; c < NPAD / 4; ++c) {
                            const float4 t = __ldcg(src + j * split_stride + c);
                            acc[4 * c] += t.x;
                            acc[4 * c + 1] += t.y;
                            acc[4 * c + 2] += t.z;
                            acc[4 * c + 3] += t.w;
                        }
                    if (n < p.N) store_column<OUT, NPAD>(p, M, n, acc);
                    if (warp == 2 && lane == 0) p.counters[nt] = 0u;   // every split of this tile has arrived
                }
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
    clock_record_end(p);
}

template <int NPAD, int OUT, bool W_MN>
cudaError_t launch_gemm_skinny(const GemmParams &p, int grid, cudaStream_t stream)
{
    auto kern = gemm_skinny_kernel<NPAD, OUT, W_MN>;
    constexpr uint32_t smem = SkinnyPlan<NPAD>::alloc_bytes;
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

// bn carries NPAD for the swap-AB entries; cluster = 0 marks them.
#define TGEMM_SKINNY_VARIANT(NPAD, OUT, BMN) \
    {NPAD, kSkinnyStages, OUT, BMN, SkinnyPlan<NPAD>::alloc_bytes, &launch_gemm_skinny<NPAD, OUT, (BMN) != 0>, 0, nullptr}

}  // namespace tgemm
