// Persistent GEMM on CTA pairs (tcgen05 cta_group::2): one 256 x 256 output
// tile per cluster of two CTAs on neighbouring SMs.
//
// Each CTA of the pair stages its own half of both operands: the leader
// (rank 0) rows [m0, m0 + 128) of A and B columns [n0, n0 + 128); the peer
// (rank 1) the next 128 rows of A and the next 128 columns of B.  The leader's
// single MMA thread issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16),
// which reads A and B from both CTAs' shared memory and writes each CTA's 128
// rows of D into that CTA's tensor memory.  Per CTA and k-block that is 32 KiB
// of operands for a 128 x 256 x 64 share of the work, against 48 KiB in the
// one-CTA kernel: a third less L2 -> SM traffic, and a 6-stage ring fits.
// Operand tiles are never multicast; every byte is loaded by the CTA that
// holds it.  The tile lifecycle is the one of tgemm_kernel.cuh.
//
// Synchronisation across the pair:
//   full[s]       leader only; the leader's producer arms it with the bytes of
//                 both CTAs, both producers' TMA loads complete on it;
//   empty[s]      in both CTAs; the leader's commit arrives on both;
//   tmem_full[b]  in both CTAs; the leader's commit arrives on both;
//   tmem_empty[b] leader only; all eight epilogue warps of the pair arrive.
// A cluster barrier after barrier initialisation and another before the
// tensor memory is freed keep either CTA from running ahead of the other.
//
// Stream-K tail (sk_units > 0).  When the tiles do not fill whole waves of
// pairs, the tiles of the last one or two waves are not dealt out whole: their
// k-block iterations are shared evenly among the pairs (StreamK in
// tgemm_sched.h).  A pair whose share covers a tile only in part writes its
// FP32 partial tile to a workspace slot and bumps that tile's arrival counter
// (one counter per CTA half); the CTA that arrives last adds the partials in
// k order -- a fixed order, independent of timing -- casts, stores C and
// resets the counter.  Nobody waits for another pair.  Splitting work by
// iterations instead of tiles is this library's choice; the pages deal whole
// tiles to blocks.
#pragma once

#include "tgemm_kernel.cuh"

namespace tgemm {

constexpr int kPairBM = 256;        // rows of a pair tile (128 per CTA)
constexpr int kPairBN = 256;        // columns of a pair tile (B split 128 + 128)

// One work item of a CTA pair: a k-block range of one tile.
struct PairWork {
    int tile;          // tile number in grouped order
    int k0, k1;        // k-blocks [k0, k1)
    bool partial;      // a stream-K segment: the tile is shared with other pairs
    bool reverse;      // run the k-blocks from k1 - 1 down to k0 (odd waves of whole tiles)
    int64_t t_sk;      // tail tile index (partial segments)
    int64_t slot;      // workspace slot (partial segments)
};

// The k-block of step j (0 .. k1 - k0 - 1) of a work item.  Whole tiles of
// odd waves run their K loop backwards: every wave of a persistent grid reads
// the same band of A rows k-block by k-block, and a band larger than what L2
// keeps is evicted in the order it was read, so a wave that starts where the
// previous one ended finds that end still in L2 instead of re-reading the
// whole band from HBM.  The sum's order changes with the direction, which
// stays fixed per configuration and shape.
__device__ __forceinline__ int work_kb(const PairWork &w, int j) { return w.reverse ? w.k1 - 1 - j : w.k0 + j; }

// The items of pair `cid` of `P`: first the segments of its stream-K share
// of the tail tiles, then whole tiles cid, cid + P, ... below dp_tiles.
// Doing the shared tiles first lets their partial-sum hand-off and final
// additions run in the epilogue warps while the whole tiles' MMAs proceed.
struct PairWorkIter {
    int next_dp, dp_tiles, P, kb, waves;
    StreamK sk;
    int64_t unit, it, end;
    bool alternate;

    __device__ PairWorkIter(const GemmParams &p, int cid, int num_pairs)
        : next_dp(cid), dp_tiles(p.dp_tiles), P(num_pairs), kb(p.num_kb), waves(0),
          sk{p.sk_tiles, p.sk_units > 0 ? p.sk_units : 1, p.num_kb}, unit(cid), it(0), end(0),
          alternate(p.k_alternate != 0)
    {
        if (p.sk_units > 0 && cid < p.sk_units) {
            it = sk.bound(cid);
            end = sk.bound(cid + 1);
        }
    }

    __device__ bool next(PairWork &w)
    {
        if (it < end) {
            const int64_t t = it / kb;
            const int64_t tile_end = (t + 1) * kb;
            const int64_t stop = end < tile_end ? end : tile_end;
            w.tile = (int)(dp_tiles + t);
            w.k0 = (int)(it - t * kb);
            w.k1 = (int)(stop - t * kb);
            w.partial = !(w.k0 == 0 && w.k1 == kb);
            w.reverse = false;
            w.t_sk = t;
            w.slot = sk.slot(unit, t);
            it = stop;
            return true;
        }
        if (next_dp < dp_tiles) {
            w.tile = next_dp;
            w.k0 = 0;
            w.k1 = kb;
            w.partial = false;
            w.reverse = alternate && (waves & 1);
            ++waves;
            next_dp += P;
            return true;
        }
        return false;
    }
};

template <int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
__global__ void __launch_bounds__(kThreads, 1) gemm_pair_kernel(const __grid_constant__ GemmParams p)
{
    static_assert(KIND == KIND_F16 || !B_MN, "FP8 and TF32 operands are K-major only");
    constexpr int kHalfN = kPairBN / 2;
    using Plan = SmemPlan<kHalfN, STAGES>;                 // A 16 KiB + B 16 KiB per stage
    constexpr uint32_t kPairStageBytes = 2 * (Plan::a_stage + Plan::b_stage);
    constexpr uint32_t kTmemCols = 512;                     // two 256-column accumulators
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
    const uint32_t rank = ptx::cluster_ctarank();           // 0 = leader, 1 = peer
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
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
    ptx::cluster_sync();          // both CTAs' barriers initialised, pair TMEM allocated
    ptx::tc_fence_after_sync();
    ptx::grid_dependency_wait();   // inputs written and outputs read by earlier kernels are settled
    clock_record_begin(p);
    ptx::launch_dependents();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(base_ptr + Plan::slot_off);

    WaitCtx wc{p.status, abort_flag, p.timeout_ns};
    wc.peer_abort = ptx::map_to_cta(abort_addr, rank ^ 1u);
    const int cluster_id = blockIdx.x >> 1;
    const int num_clusters = gridDim.x >> 1;
    bool aborted = false;

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
                batched_tile(p, w.tile, bz, tr, tc);
                const int32_t m0 = (int32_t)tr * kPairBM + 128 * (int32_t)rank;
                const int32_t n0 = (int32_t)tc * kPairBN + kHalfN * (int32_t)rank;
                const int32_t za = p.a_batched ? bz : 0, zb = p.b_batched ? bz : 0;
                for (int j = 0; j < w.k1 - w.k0; ++j) {
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, wc, SITE_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::map_to_cta(full_bar(s), 0);   // the leader's barrier
                    if (leader) ptx::mbar_arrive_expect_tx(full_bar(s), kPairStageBytes);
                    const int32_t k0 = work_kb(w, j) * KBlock<KIND>::elems;
                    ptx::tma_load_3d_pair(sA + s * Plan::a_stage, &p.tma_a, fb, k0, m0, za);
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
                // Wind down: the leader waits for the loads of both CTAs that
                // complete on its barriers (bounded; a phase the peer never
                // issued simply runs out).
                if (leader)
                    for (int t = 0; t < STAGES; ++t)
                        if (issued_mask & (1u << t))
                            wait_bounded(full_bar(t), (issued_parity >> t) & 1u, wc, SITE_DRAIN_LOADS, false);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA (leader)
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
                    // Two k-blocks in adjacent stages per pass when the second
                    // one's data is already in (one fence, one loop overhead for
                    // both): the lone issuing thread's per-k-block overhead would
                    // otherwise idle the tensor pipe.  The second stage is only
                    // tested, never waited for, so a tile's first MMAs are not
                    // held back while the ring fills.  (kb counts the steps of
                    // the item; the producer decides which k-block each is.)
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
                            ptx::mma_commit_pair(empty_bar(s + h), 0x3);   // the stage is free in both CTAs
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
                ptx::mma_commit_pair(tfull_bar(buf), 0x3);     // both halves of the accumulator ready
            }
            if (!ok) {
                aborted = true;
                ptx::mma_commit_pair(drain_bar, 0x1);
                wait_bounded(drain_bar, 0, wc, SITE_DRAIN_MMA, false);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
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
            // below synchronises them, so none may leave alone).
            if (!ptx::named_barrier_and(2, kEpiWarps * 32, got)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();

            int64_t tr, tc;
            int bz;
            batched_tile(p, w.tile, bz, tr, tc);
            ectx.z = bz;
            const int32_t row0 = (int32_t)tr * kPairBM + 128 * (int32_t)rank + 32 * q;
            const int32_t col0 = (int32_t)tc * kPairBN;
            const uint32_t t_acc = tmem_base + lane_base + buf * kPairBN;
            const uint32_t release_bar = ptx::map_to_cta(tempty_bar(buf), 0);
            if (!w.partial) {
                epilogue_drain<kPairBN, OUT>(&p.tma_c, p.M, p.N, t_acc, stage_base, cc, row0, col0, lane,
                                             [&] { ptx::mbar_arrive_cluster(release_bar); }, ectx);
                continue;
            }
            // ---- stream-K segment: FP32 partial tile into the workspace
            const int32_t prow = (int32_t)(w.slot * kPairBM) + 128 * (int32_t)rank + 32 * q;
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
                const uint32_t prev = atomicAdd(&p.counters[2 * w.t_sk + rank], 1u);
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
                        const float4 *src = reinterpret_cast<const float4 *>(
                            p.partials + ((sk.slot(u, w.t_sk) * kPairBM + warp_row + sub_row) * kPairBN + c * kCols) +
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
                if (ew == 0 && lane == 0) p.counters[2 * w.t_sk + rank] = 0u;   // ready for the next call
            }
        }
        if (lane == 0) ptx::bulk_wait_group_all();
        __syncwarp();
    }

    if (aborted || *abort_flag) {
        // After a timeout, give copies issued by either CTA of the pair (their
        // completion may be signalled in the other CTA) time to land before
        // the shared memory is released: about 200 us, far above a TMA round trip.
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::cluster_sync();          // neither CTA frees TMEM or exits while its partner still works
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    clock_record_end(p);
}

template <int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
cudaError_t launch_gemm_pair(const GemmParams &p, int grid, cudaStream_t stream)
{
    auto kern = gemm_pair_kernel<STAGES, OUT, B_MN, KIND>;
    constexpr uint32_t smem = SmemPlan<kPairBN / 2, STAGES>::alloc_bytes;
    static std::atomic<unsigned long long> smem_set{0};
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
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

// Number of CTA pairs of this kernel that can be resident at once.
template <int STAGES, int OUT, bool B_MN, int KIND = KIND_F16>
int max_active_pairs()
{
    auto kern = gemm_pair_kernel<STAGES, OUT, B_MN, KIND>;
    constexpr uint32_t smem = SmemPlan<kPairBN / 2, STAGES>::alloc_bytes;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
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

#define TGEMM_PAIR_VARIANT(ST, OUT, BMN)                                                              \
    {256, ST, OUT, BMN, SmemPlan<kPairBN / 2, ST>::alloc_bytes, &launch_gemm_pair<ST, OUT, (BMN) != 0>, \
     2, &max_active_pairs<ST, OUT, (BMN) != 0>}
#define TGEMM_PAIR_VARIANT_KIND(ST, OUT, KIND)                                                            \
    {256, ST, OUT, 0, SmemPlan<kPairBN / 2, ST>::alloc_bytes, &launch_gemm_pair<ST, OUT, false, KIND>, 2, \
     &max_active_pairs<ST, OUT, false, KIND>, KIND}

}  // namespace tgemm
