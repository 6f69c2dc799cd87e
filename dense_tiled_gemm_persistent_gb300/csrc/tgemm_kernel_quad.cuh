// Persistent GEMM on clusters of two CTA pairs ("quads"): one 256 x 512
// output block per cluster of four CTAs, pair q (ranks 2q, 2q + 1) computing
// the 256 x 256 tile in columns [n0 + 256 q, n0 + 256 q + 256).
//
// Both pairs need the same 256 rows of A, so each A half-tile is fetched once
// for the two pairs: CTA 2q + r (r = rank in its pair) loads rows
// [m0 + 128 r + 64 q, + 64) of the k-block and multicasts them to CTAs r and
// r + 2, which each receive the full 128 rows of their half from the two
// loads.  B is loaded by each CTA for itself, as in the pair kernel.  Per CTA
// and k-block that is 24 KiB of TMA requests instead of 32 KiB: a quarter
// less L2 -> SM traffic and TMA request rate for the same tensor work, which
// matters where rows of A and B are not 128-byte aligned (every box row then
// straddles two cache lines) and for the energy of a power-capped GEMM.
// Multicast stays inside one GPU's memory.
//
// Synchronisation (per stage s, per accumulator buffer b):
//   full[s]       in each pair leader; armed with the pair's 64 KiB, completed by
//                 the pair's B loads and by the A loads of both pairs (a
//                 multicast load signals each destination's pair leader);
//   empty[s]      in all four CTAs, count 2: both pair leaders' MMA commits
//                 arrive on every CTA, since a stage is refilled only when
//                 neither pair still reads it (its A rows come from both);
//   tmem_full[b]  in both CTAs of a pair; that pair's leader commits;
//   tmem_empty[b] in each pair leader; the pair's eight epilogue warps arrive.
// Every wait is bounded (tgemm_wait.cuh); a timeout raises the abort flag in
// all four CTAs, which then wind down as the pair kernel does.  When the
// tile columns are odd the second pair of the last block column computes a
// tile past N (its B reads zeros, its stores are skipped) so that it still
// feeds its partner's A.
//
// Stream-K tail (sk_units > 0), as in the pair kernel but with 256 x 512
// blocks as the shared items: both pairs of a quad run the same k-range of
// the same block (they share its A rows), each writes the FP32 partial of
// its own tile, and per tile half the last arriving CTA adds the partials
// in k order (quad_stream_k_segment).
#pragma once

#include "tgemm_kernel_pair.cuh"

namespace tgemm {

constexpr int kQuadBN = 2 * kPairBN;    // columns of a quad block
constexpr int kQuadTiles = 2;          // pair tiles per quad block

// A stream-K segment of the quad kernel, in the four epilogue warps of one
// CTA: the CTA's FP32 partial of its 128-row half of tile jt of a 256 x 512
// block goes to a workspace slot (TMA stores), the tile half's arrival
// counter is bumped, and the CTA that brings the last segment adds all of
// them in k order (unit u0, u0 + 1, ...: fixed, so results do not depend on
// timing), applies the fused epilogue, casts, stores C and resets the
// counter.  Slot s of a unit holds tile jt at workspace rows (2 s + jt) * 256;
// the counter of tile jt's half `rank` is (2 t_sk + jt) * 2 + rank.  The pair
// kernel does the same step inline for one tile per item; calling a shared
// function from it changed its code generation (228 instead of 226
// registers) and made whole-tile launches 1-1.5 % slower on 8192^3, 4096^3
// and 4096 x 3072 x 5000 (same GB300, alternating builds), so the two copies
// stay separate.
template <int OUT>
__device__ __forceinline__ void quad_stream_k_segment(const GemmParams &p, const PairWork &w, int jt, uint32_t rank,
                                                      int q, int ew, int lane, int32_t row0, int32_t col0, int bz,
                                                      uint32_t t_acc, uint32_t stage_base, uint32_t &cc,
                                                      uint32_t release_bar, volatile int *last_flag, EpiCtx &ectx,
                                                      EpiCtx &raw)
{
    const int64_t counter = (w.t_sk * kQuadTiles + jt) * 2 + rank;
    const int32_t prow = (int32_t)((w.slot * kQuadTiles + jt) * kPairBM) + 128 * (int32_t)rank + 32 * q;
    epilogue_drain<kPairBN, OUT_F32>(&p.tma_ws, INT32_MAX, kPairBN, t_acc, stage_base, cc, prow, 0, lane,
                                     [&] { ptx::mbar_arrive_cluster(release_bar); }, raw);
    if (lane == 0) {
        ptx::bulk_wait_group_all();          // this warp's partial rows are written
        ptx::fence_proxy_async_global();
    }
    __syncwarp();
    __threadfence();
    const StreamK sk{p.sk_tiles, p.sk_units, p.num_kb};
    const int64_t first = w.t_sk * p.num_kb, stop = first + p.num_kb;
    const int64_t u0 = sk.unit_of(first);
    ptx::named_barrier(1, kEpiWarps * 32);
    if (ew == 0 && lane == 0) {
        uint32_t segs = 0;
        for (int64_t u = u0; u < sk.sk_units && sk.bound(u) < stop; ++u) ++segs;
        const uint32_t prev = atomicAdd(&p.counters[counter], 1u);
        *last_flag = (prev + 1 == segs) ? 1 : 0;
    }
    ptx::named_barrier(1, kEpiWarps * 32);
    if (*last_flag) {
        // Every segment of this tile half is in: add them in k order.
        __threadfence();
        // Column-parallel over this warp's 32 rows: per store chunk (32
        // FP32 or 64 16-bit columns) each lane owns 4 columns of a row,
        // so every load of the warp reads whole row segments.  The sums
        // go straight into the warp's swizzled staging block, which a
        // TMA store then writes to C.
        constexpr int kCols = OUT == OUT_F32 ? 32 : 64;
        constexpr int kLanesPerRow = kCols / 4;
        constexpr int kRowsPerPass = 32 / kLanesPerRow;
        constexpr int kPasses = 32 / kRowsPerPass;
        const int sub_row = lane / kLanesPerRow, col4 = lane % kLanesPerRow;
        int64_t u_end = u0;
        while (u_end < sk.sk_units && sk.bound(u_end) < stop) ++u_end;
        const int64_t warp_row = 128 * (int64_t)rank + 32 * q;       // first row of this warp in the tile
#pragma unroll 1
        for (int c = 0; c < kPairBN / kCols; ++c) {
            float4 acc[kPasses];
#pragma unroll
            for (int i = 0; i < kPasses; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int64_t u = u0; u < u_end; ++u) {                    // k order: unit u0, u0 + 1, ...
                const int64_t prow_u = (sk.slot(u, w.t_sk) * kQuadTiles + jt) * kPairBM + warp_row + sub_row;
                const float4 *src = reinterpret_cast<const float4 *>(p.partials + (prow_u * kPairBN + c * kCols) +
                                                                     col4 * 4);
                float4 t[kPasses];
#pragma unroll
                for (int i = 0; i < kPasses; ++i) t[i] = __ldcg(src + (int64_t)i * kRowsPerPass * (kPairBN / 4));
#pragma unroll
                for (int i = 0; i < kPasses; ++i) {
                    acc[i].x += t[i].x;
                    acc[i].y += t[i].y;
                    acc[i].z += t[i].z;
                    acc[i].w += t[i].w;
                }
            }
            const uint32_t sbuf = stage_base + (cc & 1u) * kStageCBytes;
            if (lane == 0) ptx::bulk_wait_group_read<1>();
            __syncwarp();
            const bool fused = (p.epi & 1) != 0;
            const bool with_cin = fused && (p.epi & 2) && fetch_cin(ectx, sbuf, col0 + c * kCols, row0, lane);
            const int64_t col = (int64_t)col0 + c * kCols + col4 * 4;
            const EpiScalars es = EpiScalars::of(p);
#pragma unroll
            for (int i = 0; i < kPasses; ++i) {
                const uint32_t r = (uint32_t)(i * kRowsPerPass + sub_row);
                if constexpr (OUT == OUT_F32) {
                    const uint32_t addr = sbuf + r * 128 + (((uint32_t)col4 ^ (r & 7)) << 4);
                    if (fused) {
                        float4 ci = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (with_cin) ci = ptx::ld_shared_v4(addr);
                        acc[i].x = epi_value(es, acc[i].x, ci.x, col);
                        acc[i].y = epi_value(es, acc[i].y, ci.y, col + 1);
                        acc[i].z = epi_value(es, acc[i].z, ci.z, col + 2);
                        acc[i].w = epi_value(es, acc[i].w, ci.w, col + 3);
                    }
                    ptx::st_shared_v4(addr, __float_as_uint(acc[i].x), __float_as_uint(acc[i].y),
                                      __float_as_uint(acc[i].z), __float_as_uint(acc[i].w));
                } else {
                    const uint32_t addr = sbuf + r * 128 + ((((uint32_t)col4 >> 1) ^ (r & 7)) << 4) + (col4 & 1) * 8;
                    if (fused) {
                        float2 c0 = make_float2(0.f, 0.f), c1 = make_float2(0.f, 0.f);
                        if (with_cin) {
                            uint32_t q0, q1;
                            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(q0), "=r"(q1) : "r"(addr) : "memory");
                            c0 = unpack_out(q0, OUT);
                            c1 = unpack_out(q1, OUT);
                        }
                        acc[i].x = epi_value(es, acc[i].x, c0.x, col);
                        acc[i].y = epi_value(es, acc[i].y, c0.y, col + 1);
                        acc[i].z = epi_value(es, acc[i].z, c1.x, col + 2);
                        acc[i].w = epi_value(es, acc[i].w, c1.y, col + 3);
                    }
                    const uint32_t a0 = pack_out(acc[i].x, acc[i].y, OUT);
                    const uint32_t a1 = pack_out(acc[i].z, acc[i].w, OUT);
                    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a0), "r"(a1) : "memory");
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int32_t x = col0 + c * kCols;
                if (x < p.N && row0 < p.M) ptx::tma_store_3d(&p.tma_c, sbuf, x, row0, bz);
                ptx::bulk_commit_group();
            }
            ++cc;
        }
        if (ew == 0 && lane == 0) p.counters[counter] = 0u;   // ready for the next call
    }
}


template <int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
__global__ void __launch_bounds__(kThreads, 1) gemm_quad_kernel(const __grid_constant__ GemmParams p)
{
    static_assert(KIND == KIND_F16 || !B_MN, "FP8 and TF32 operands are K-major only");
    constexpr int kHalfN = kPairBN / 2;
    using Plan = SmemPlan<kHalfN, STAGES>;                 // A 16 KiB + B 16 KiB per stage
    constexpr uint32_t kPairStageBytes = 2 * (Plan::a_stage + Plan::b_stage);
    constexpr uint32_t kAHalfBytes = Plan::a_stage / 2;     // 64 rows of A
    constexpr uint32_t kTmemCols = 512;
    static_assert(Plan::alloc_bytes <= 232448, "shared memory plan exceeds 227 KiB");

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
    const uint32_t abort_addr = base + Plan::abort_off;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_ptr + Plan::abort_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();          // 0..3
    const uint32_t q = crank >> 1;                          // pair of the quad
    const uint32_t rank = crank & 1u;                       // rank in the pair
    const uint32_t pair_leader = 2u * q;
    const bool leader = rank == 0;
    const uint16_t pair_mask = (uint16_t)(0x3u << (2u * q));
    const uint16_t a_mask = (uint16_t)((1u << rank) | (1u << (rank + 2u)));   // this A half's two holders

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 2);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), 2 * kEpiWarps);
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
        ptx::tmem_alloc_pair(slot, kTmemCols);
        ptx::tmem_relinquish_pair();
        ptx::tc_fence_before_sync();
    }
    __syncthreads();
    ptx::cluster_sync();          // all four CTAs' barriers initialised, both pairs' TMEM allocated
    ptx::tc_fence_after_sync();
    ptx::grid_dependency_wait();   // inputs written and outputs read by earlier kernels are settled
    clock_record_begin(p);
    ptx::launch_dependents();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(base_ptr + Plan::slot_off);

    WaitCtx wc{p.status, abort_flag, p.timeout_ns};
    wc.peer_mask = 0xFu & ~(1u << crank);
    wc.abort_local = abort_addr;
    const int cluster_id = blockIdx.x >> 2;
    const int num_clusters = gridDim.x >> 2;
    bool aborted = false;

    // Block number -> (batch, block row, this pair's tile column).
    auto block_coord = [&](int blk, int &bz, int64_t &tr, int64_t &tc) {
        int32_t r, cq;
        bz = blk / p.tiles_per_batch;
        grouped_tile32(p.tiles_m, p.tiles_n, p.group_m, blk - bz * p.tiles_per_batch, r, cq);
        tr = r;
        tc = 2 * (int64_t)cq + q;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            PairWorkIter items(p, cluster_id, num_clusters);
            PairWork w;
            while (ok && items.next(w)) {
                int64_t tr, tc;
                int bz;
                block_coord(w.tile, bz, tr, tc);
                const int32_t m0 = (int32_t)tr * kPairBM + 128 * (int32_t)rank + 64 * (int32_t)q;
                const int32_t n0 = (int32_t)tc * kPairBN + kHalfN * (int32_t)rank;
                const int32_t za = p.a_batched ? bz : 0, zb = p.b_batched ? bz : 0;
                for (int j = 0; j < w.k1 - w.k0; ++j) {
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, wc, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::map_to_cta(full_bar(s), pair_leader);
                    if (leader) ptx::mbar_arrive_expect_tx(full_bar(s), kPairStageBytes);
                    const int32_t k0 = work_kb(w, j) * KBlock<KIND>::elems;
                    ptx::tma_load_3d_pair_mc(sA + s * Plan::a_stage + q * kAHalfBytes, &p.tma_a, fb, k0, m0, za,
                                             a_mask);
                    if (B_MN) {
#pragma unroll
                        for (int j = 0; j < kHalfN / 64; ++j)
                            ptx::tma_load_3d_pair(sB + s * Plan::b_stage + j * (kBK * 128), &p.tma_b, fb,
                                                  n0 + 64 * j, k0, zb);
                    } else {
                        ptx::tma_load_3d_pair(sB + s * Plan::b_stage, &p.tma_b, fb, k0, n0, zb);
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
                aborted = true;
                if (leader)
                    for (int t = 0; t < STAGES; ++t)
                        if (issued_mask & (1u << t))
                            wait_bounded(full_bar(t), (issued_parity >> t) & 1u, wc, SITE_DRAIN_LOADS, false);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA (pair leaders)
        if (lane == 0 && leader) {
            const uint64_t kDescB = B_MN ? kDescMNMajor : kDescKMajor;
            int s = 0;
            uint32_t ph = 0;
            uint32_t local = 0;
            bool ok = true;
            PairWorkIter items(p, cluster_id, num_clusters);
            PairWork w;
            for (; ok && items.next(w); ++local) {
                const uint32_t buf = local & 1u;
                const uint32_t bph = (local >> 1) & 1u;
                if (!wait_bounded(tempty_bar(buf), bph ^ 1u, wc, SITE_MMA_TMEM_EMPTY)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * kPairBN;
                for (int kb = w.k0; kb < w.k1;) {
                    // two k-blocks per pass when the second stage is already full
                    if (!wait_bounded(full_bar(s), ph, wc, SITE_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    const int n =
                        (kb + 1 < w.k1 && s + 1 < STAGES && ptx::mbar_test_wait(full_bar(s + 1), ph)) ? 2 : 1;
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < n) {
                            const uint32_t a_addr = sA + (s + h) * Plan::a_stage;
                            const uint32_t b_addr = sB + (s + h) * Plan::b_stage;
#pragma unroll
                            for (int k = 0; k < kBK / kUmmaK; ++k) {
                                const uint64_t ad = desc_at(kDescKMajor, a_addr + k * (kUmmaK * 2));
                                const uint64_t bd =
                                    desc_at(kDescB, b_addr + (B_MN ? k * (kUmmaK * 128) : k * (kUmmaK * 2)));
                                mma_issue<KIND, true>(d_tmem, ad, bd, p.idesc, (kb + h > w.k0 || k > 0) ? 1u : 0u);
                            }
                            ptx::mma_commit_pair(empty_bar(s + h), 0xF);   // the stage is free for this pair, in all four CTAs
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
                ptx::mma_commit_pair(tfull_bar(buf), pair_mask);    // this pair's accumulator is ready
            }
            if (!ok) {
                aborted = true;
                ptx::mma_commit_pair(drain_bar, (uint16_t)(1u << crank));
                wait_bounded(drain_bar, 0, wc, SITE_DRAIN_MMA, false);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;
        const int qw = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * qw) << 16;
        const uint32_t stage_base = sC + ew * 2 * kStageCBytes;
        volatile int *last_flag = reinterpret_cast<volatile int *>(base_ptr + Plan::flag_off);
        EpiCtx ectx{&p, drain_bar + 8u * (1 + ew), 0u, wc};
        EpiCtx raw{nullptr, 0u, 0u, wc};                 // stream-K partials: raw FP32
        uint32_t local = 0, cc = 0;
        PairWorkIter items(p, cluster_id, num_clusters);
        PairWork w;
        for (; items.next(w); ++local) {
            const uint32_t buf = local & 1u;
            const uint32_t bph = (local >> 1) & 1u;
            const bool got = wait_bounded(tfull_bar(buf), bph, wc, SITE_EPI_TMEM_FULL);
            // The four epilogue warps decide together (the stream-K hand-off
            // synchronises them, so none may leave alone).
            if (!ptx::named_barrier_and(2, kEpiWarps * 32, got)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            int64_t tr, tc;
            int bz;
            block_coord(w.tile, bz, tr, tc);
            ectx.z = bz;
            const int32_t row0 = (int32_t)tr * kPairBM + 128 * (int32_t)rank + 32 * qw;
            const int32_t col0 = (int32_t)tc * kPairBN;
            const uint32_t t_acc = tmem_base + lane_base + buf * kPairBN;
            const uint32_t release_bar = ptx::map_to_cta(tempty_bar(buf), pair_leader);
            if (!w.partial) {
                epilogue_drain<kPairBN, OUT>(&p.tma_c, p.M, p.N, t_acc, stage_base, cc, row0, col0, lane,
                                             [&] { ptx::mbar_arrive_cluster(release_bar); }, ectx);
                continue;
            }
            // stream-K segment of this pair's tile (tile q of the block)
            quad_stream_k_segment<OUT>(p, w, (int)q, rank, qw, ew, lane, row0, col0, bz, t_acc, stage_base, cc,
                                     release_bar, last_flag, ectx, raw);
        }
        if (lane == 0) ptx::bulk_wait_group_all();
        __syncwarp();
    }

    if (aborted || *abort_flag) {
        // copies issued by any CTA of the quad may land in this one: let them settle
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::cluster_sync();          // no CTA frees TMEM or exits while another still works
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    clock_record_end(p);
}

template <int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
cudaError_t launch_gemm_quad(const GemmParams &p, int grid, cudaStream_t stream)
{
    auto kern = gemm_quad_kernel<STAGES, OUT, B_MN, KIND>;
    constexpr uint32_t smem = SmemPlan<kPairBN / 2, STAGES>::alloc_bytes;
    static std::atomic<unsigned long long> smem_set{0};
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see ptx::grid_dependency_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Number of quads (clusters of four) of this kernel that can be resident at once.
template <int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
int max_active_quads()
{
    auto kern = gemm_quad_kernel<STAGES, OUT, B_MN, KIND>;
    constexpr uint32_t smem = SmemPlan<kPairBN / 2, STAGES>::alloc_bytes;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Variant table entries: cluster 4 = quad.
#define TGEMM_QUAD_VARIANT(ST, OUT, BMN)                                                              \
    {256, ST, OUT, BMN, SmemPlan<kPairBN / 2, ST>::alloc_bytes, &launch_gemm_quad<ST, OUT, (BMN) != 0>, \
     4, &max_active_quads<ST, OUT, (BMN) != 0>}
#define TGEMM_QUAD_VARIANT_KIND(ST, OUT, KIND)                                                            \
    {256, ST, OUT, 0, SmemPlan<kPairBN / 2, ST>::alloc_bytes, &launch_gemm_quad<ST, OUT, false, KIND>, 4, \
     &max_active_quads<ST, OUT, false, KIND>, KIND}

}  // namespace tgemm
