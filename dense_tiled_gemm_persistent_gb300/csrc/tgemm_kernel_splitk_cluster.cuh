// Skinny GEMM with split-K reduced inside a thread-block cluster.
//
// Same swap-AB formulation as tgemm_kernel_skinny.cuh (C^T = B^T * A^T: 128
// weight rows on the MMA's M side, the <= 128 rows of A padded to NPAD on its N
// side), but the S CTAs that split the K loop of one 128-column tile of C
// form one cluster and add their partial sums through distributed shared
// memory instead of a global workspace:
//
//   1. every CTA runs its K range through a STAGES-deep TMA ring and reads
//      its 128 x NPAD FP32 partial from tensor memory into registers, one
//      32-row quarter per epilogue warp;
//   2. quarter q is reduced by rank q mod min(S, 4), its owner (so up to
//      four CTAs of the cluster reduce and store at once, each receiving a
//      quarter of what one leader would); once an owner's MMAs are done
//      reading its ring, its MMA thread arrives on a "ring free" mbarrier in
//      each other rank;
//   3. the other ranks' warps q wait for that and send their quarter into
//      the owner's ring with st.async, each store counting its 16 bytes on
//      the owner's "partials" mbarrier (which expects the bytes of every
//      quarter it owns from every other rank);
//   4. the owner waits for those bytes;
//   5. its warp q adds the partials of quarter q in rank order 0, 1, ...,
//      S-1 (fixed, so results do not depend on timing), applies the fused
//      epilogue, casts with round-to-nearest-even and stores from registers
//      (32 consecutive columns of each row of C per warp).
//
// Measured on 16 x 4096 x 4096 (four ranks), the leader-only reduction
// spent 0.4 us receiving 24 KiB through distributed shared memory, 0.3 us
// summing and 0.25 us staging and storing the tile.
//
// No CTA waits for the whole cluster on the way: a cluster barrier's
// release/acquire costs about a microsecond here, two of them a tenth of a
// 32 MiB projection.  The barrier halves at start and exit only order the
// mbarrier set-up and keep every CTA's shared memory alive while others may
// write into it.  After a fault the ranks still send their (meaningless)
// partials, so an owner never waits for bytes that will not come; the
// status word reports the fault.
// No device memory besides A, B and C is touched, no atomics, no counters.
// S is limited by the cluster size (8) and, conservatively, by a ring
// holding S-1 whole partials.
//
// RING_KB is the operand ring's budget.  216 KiB keeps one CTA per SM with
// the most weight bytes in flight; 108 KiB lets two CTAs share an SM, so the
// CTAs of the next launch can be resident (prologue done, waiting on
// griddepcontrol.wait) while this one streams its weights.
#pragma once

#include "tgemm_kernel_skinny.cuh"

namespace tgemm {

constexpr int kMaxClusterSplits = 8;

template <int NPAD, int RING_KB = 216>
struct ClusterSplitPlan {
    static constexpr uint32_t w_stage = kSkinnyRows * kBK * 2;
    static constexpr uint32_t x_stage = NPAD * kBK * 2;
    static constexpr uint32_t stage_bytes = w_stage + x_stage;
    // 216 KiB: 12, 10, 9 stages for NPAD 16, 32, 64 (6 for 128); 108 KiB: 6, 5, 4
    static constexpr int stages = (int)((RING_KB * 1024u) / stage_bytes);
    static constexpr int ctas_per_sm = RING_KB <= 108 ? 2 : 1;
    static constexpr uint32_t w_off = 0;
    static constexpr uint32_t x_off = w_off + stages * w_stage;
    static constexpr uint32_t bar_off = x_off + stages * x_stage;
    // full[S], empty[S], tmem_full, drain, partials, drain 2, ring free[4]
    static constexpr uint32_t n_bars = 2 * stages + 8;
    static constexpr uint32_t slot_off = bar_off + 8 * n_bars;
    static constexpr uint32_t abort_off = slot_off + 4;
    static constexpr uint32_t bytes = abort_off + 4;
    static constexpr uint32_t alloc_bytes = bytes + 1024;
    static constexpr uint32_t partial_bytes = kSkinnyRows * NPAD * 4;   // one CTA's 128 x NPAD partial
    static constexpr uint32_t quarter_bytes = partial_bytes / 4;         // its 32 rows of one epilogue warp
    // An owner's ring (from offset 0) receives, for each quarter it owns (at
    // most two), the other ranks' partials of it; bounded here, more loosely,
    // by S-1 whole partials.
    static constexpr int max_splits_by_ring = 1 + (int)((stages * stage_bytes) / partial_bytes);
    static constexpr int max_splits = max_splits_by_ring < kMaxClusterSplits ? max_splits_by_ring : kMaxClusterSplits;
    // The slots an owner's ring holds at S splits: S per quarter it owns (at
    // most 4 / min(S, 4), rounded up).
    static constexpr bool slots_fit(int s)
    {
        return s > max_splits ||
               (uint32_t)((4 + (s < 4 ? s : 4) - 1) / (s < 4 ? s : 4) * s) * quarter_bytes <= stages * stage_bytes;
    }
    static constexpr bool all_slots_fit(int s = 2) { return s > kMaxClusterSplits || (slots_fit(s) && all_slots_fit(s + 1)); }
    static_assert(all_slots_fit(), "an owner's ring must hold the partials of its quarters");
};

template <int NPAD, int OUT, bool W_MN, int RING_KB, int KIND = KIND_F16>
__global__ void __launch_bounds__(kThreads, ClusterSplitPlan<NPAD, RING_KB>::ctas_per_sm)
    gemm_splitk_cluster_kernel(const __grid_constant__ GemmParams p)
{
    using Plan = ClusterSplitPlan<NPAD, RING_KB>;
    constexpr int S = Plan::stages;
    // FP16/BF16 (kind::f16, 64 elements per 128-byte k-block row) or FP8
    // (kind::f8f6f4, 128 elements): the same bytes per stage and per MMA
    static_assert(KIND == KIND_F16 || (KIND == KIND_F8 && !W_MN), "FP8 weights are K-major only");
    constexpr int kKE = KBlock<KIND>::elems;
    constexpr uint32_t kTmemCols = SkinnyAcc<NPAD>::tmem_cols;
    static_assert(Plan::alloc_bytes <= 232448, "shared memory plan exceeds 227 KiB");
    static_assert(Plan::ctas_per_sm == 1 || Plan::alloc_bytes <= 232448 / 2 - 1024,
                  "two CTAs of this plan must fit one SM");

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
    const uint32_t drain_bar = bar + 8u * (2 * S + 1);
    const uint32_t part_bar = bar + 8u * (2 * S + 2);   // owners: the other ranks' partials have arrived
    const uint32_t drain2_bar = bar + 8u * (2 * S + 3); // the second MMA issuer's wind-down
    auto free_bar = [&](int o) { return bar + 8u * (2 * S + 4 + o); };   // owner o's ring may be filled
    const uint32_t slot = base + Plan::slot_off;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_ptr + Plan::abort_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int splits = p.splits;                   // = cluster size
    const uint32_t rank = ptx::cluster_ctarank();  // = split index
    const int nt = blockIdx.x / splits;
    const int kb0 = (int)((int64_t)rank * p.num_kb / splits);
    const int kb1 = (int)((int64_t)(rank + 1) * p.num_kb / splits);
    const int32_t n0 = nt * kSkinnyRows;
    // Quarter q of the tile (weight rows 32q..32q+31, epilogue warp q) is
    // reduced and stored by rank q mod min(S, 4), its owner.
    const int owners = splits < 4 ? splits : 4;
    int owned = 0;                                  // quarters this rank owns
    for (int q = 0; q < 4; ++q) owned += (q % owners == (int)rank) ? 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        ptx::mbar_init(tfull_bar, kSkinnyIssuers);
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(drain2_bar, 1);
        for (int o = 0; o < 4; ++o) ptx::mbar_init(free_bar(o), 1);
        ptx::mbar_init(part_bar, 1);
        if (owned > 0 && splits > 1)
            ptx::mbar_arrive_expect_tx(part_bar, (uint32_t)(owned * (splits - 1)) * Plan::quarter_bytes);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&p.tma_a);
        ptx::prefetch_tensormap(&p.tma_b);
        prefetch_weights_l2<W_MN, kKE>(&p.tma_b, n0, kb0, kb1, p.prefetch_kb);
    }
    if (warp == 1) {
        ptx::tmem_alloc(slot, kTmemCols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before_sync();
    }
    __syncthreads();
    ptx::cluster_arrive_relaxed();   // this CTA's barriers are initialised (waited on before any remote access)
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(base_ptr + Plan::slot_off);
    const WaitCtx wc{p.status, abort_flag, p.timeout_ns};
    ptx::grid_dependency_wait();   // inputs written and outputs read by earlier kernels are settled
    clock_record_begin(p);
    // The next launch on the stream may start its prologue (and weight
    // prefetch) at once, or -- late_trigger -- once every CTA has issued its
    // last load (the first call in a CTA counts; the later ones in the other
    // roles are no-ops, kept so that every path reaches one).
    if (!p.late_trigger) ptx::launch_dependents();

    float v[NPAD];
#pragma unroll
    for (int m = 0; m < NPAD; ++m) v[m] = 0.f;
    bool have = false;

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
                ptx::mbar_arrive_expect_tx(fb, Plan::stage_bytes);
                const int32_t k0 = kb * kKE;
                if (W_MN) {
#pragma unroll
                    for (int j = 0; j < kSkinnyRows / 64; ++j)
                        ptx::tma_load_2d(sW + s * Plan::w_stage + j * (kBK * 128), &p.tma_b, fb, n0 + 64 * j, k0);
                } else {
                    ptx::tma_load_2d(sW + s * Plan::w_stage, &p.tma_b, fb, k0, n0);
                }
                ptx::tma_load_2d(sX + s * Plan::x_stage, &p.tma_a, fb, k0, 0);
                if (p.late_trigger && kb + 1 == kb1) ptx::launch_dependents();
                issued_mask |= 1u << s;
                issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (p.late_trigger) ptx::launch_dependents();
            if (!ok)
                for (int t = 0; t < S; ++t)
                    if (issued_mask & (1u << t))
                        wait_bounded(full_bar(t), (issued_parity >> t) & 1u, wc, SITE_DRAIN_LOADS, false);
        }
        __syncwarp();
        if (p.late_trigger) ptx::launch_dependents();
        ptx::cluster_wait();   // every CTA's barriers are initialised (the other roles wait before their loops)
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA, first issuer
        // Every CTA's barriers are initialised before the first remote
        // access.  The MMA and epilogue warps take that wait now, where it
        // overlaps the first loads, instead of after the K loop; the
        // producer after its loop, so that its first loads go out at once.
        ptx::cluster_wait();
        if (lane == 0) {
            // An owner's ring is reused for the partials of the other ranks:
            // once every MMA of this CTA (both issuers) is done reading it
            // (tfull, or the drain after a fault), the ranks that send to
            // this one may fill it.  A relaxed arrive is enough: the hazard
            // is write-after-read, the reads are done before the arrive is
            // issued and no write is issued before a rank has seen it.
            if (skinny_mma_role<NPAD, W_MN, S, Plan::w_stage, Plan::x_stage, KIND>(0, sW, sX, bar, tfull_bar, drain_bar,
                                                                             kb0, kb1, tmem_base, p.idesc, wc))
                wait_bounded(tfull_bar, 0, wc, SITE_MMA_FULL, false);
            if ((int)rank < owners)
                for (int r = 0; r < splits; ++r)
                    if (r != (int)rank)
                        ptx::mbar_arrive_remote_relaxed(ptx::map_to_cta(free_bar(rank), (uint32_t)r));
        }
        __syncwarp();
    } else {
        // -------------------------------------------------- epilogue: TMEM -> registers
        ptx::cluster_wait();
        if (warp == 2) {   // the second MMA issuer first
            if (lane == 0)
                skinny_mma_role<NPAD, W_MN, S, Plan::w_stage, Plan::x_stage, KIND>(1, sW, sX, bar, tfull_bar, drain2_bar,
                                                                             kb0, kb1, tmem_base, p.idesc, wc);
            __syncwarp();
        }
        const int q = warp & 3;
        const bool got = wait_bounded(tfull_bar, 0, wc, SITE_EPI_TMEM_FULL);
        if (__all_sync(0xffffffffu, got)) {
            ptx::tc_fence_after_sync();
            load_skinny_acc<NPAD>(tmem_base + ((uint32_t)(32 * q) << 16), kb1 - kb0, v);
            have = true;
        }
    }

    const bool epi = warp >= 2;
    const int q = warp & 3;                          // quarter of the tile (epilogue warps)
    const int owner = q % owners;
    // Slot of quarter q's partial from rank `from` (the owner's own
    // included) in its owner's ring: the owner's quarters in order, then the
    // ranks in order; inside a slot, chunk c (4 floats) of row l at
    // c * 512 + l * 16, so the 32 lanes of a warp touch 512 consecutive bytes.
    auto slot_addr = [&](int from) {
        const int idx = (q / owners) * splits + from;
        return sW + (uint32_t)idx * Plan::quarter_bytes + (uint32_t)lane * 16u;
    };
    bool received = true;
    if (splits > 1) {
        if (epi && owner != (int)rank) {
            wait_bounded(free_bar(owner), 0, wc, SITE_CLUSTER_EXCHANGE, false);
            const uint32_t dst = ptx::map_to_cta(slot_addr((int)rank), (uint32_t)owner);
            const uint32_t owner_bar = ptx::map_to_cta(part_bar, (uint32_t)owner);
#pragma unroll
            for (int c = 0; c < NPAD / 4; ++c)
                ptx::st_async_v4(dst + c * 512u, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3], owner_bar);
        }
        if (epi && owner == (int)rank) received = wait_bounded(part_bar, 0, wc, SITE_CLUSTER_EXCHANGE, false);
    }
    // Each owning warp decides for its quarter (all its lanes together).
    const bool go = epi && owner == (int)rank && __all_sync(0xffffffffu, have && received && *abort_flag == 0);
    if (go && splits > 1) {
        // Rank order 0, 1, ..., S-1 (fixed, so results do not depend on
        // timing): the owner's own partial goes to its slot first, then the
        // slots are added in place, one rank at a time.  (Keeping the own
        // partial in registers and reading the other slots all at once was
        // slower at 16 columns, 0.48 against 0.32 us, and spilled at 128.)
        const uint32_t own = slot_addr((int)rank);
#pragma unroll
        for (int c = 0; c < NPAD / 4; ++c)
            ptx::st_shared_v4(own + c * 512u, __float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                              __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
        {
            const uint32_t src = slot_addr(0);
#pragma unroll
            for (int c = 0; c < NPAD / 4; ++c) {
                const float4 t = ptx::ld_shared_v4(src + c * 512u);
                v[4 * c] = t.x;
                v[4 * c + 1] = t.y;
                v[4 * c + 2] = t.z;
                v[4 * c + 3] = t.w;
            }
        }
        for (int r = 1; r < splits; ++r) {
            const uint32_t src = slot_addr(r);
#pragma unroll
            for (int c = 0; c < NPAD / 4; ++c) {
                const float4 t = ptx::ld_shared_v4(src + c * 512u);
                v[4 * c] += t.x;
                v[4 * c + 1] += t.y;
                v[4 * c + 2] += t.z;
                v[4 * c + 3] += t.w;
            }
        }
    }
    if (go) {
        // The fused epilogue and the stores straight from registers: for
        // each row of C the warp writes 32 consecutive columns.
        const int64_t n = (int64_t)n0 + 32 * q + lane;
        if (n < p.N) store_column<OUT, NPAD>(p, p.M < NPAD ? (int)p.M : NPAD, n, v);
    }

    // The other roles' copies of the trigger, after the exchange and off
    // its path.
    if (p.late_trigger && warp != 0) ptx::launch_dependents();

    // No CTA leaves while another may still write into its shared memory:
    // an owner arrives once every partial it expects has landed, the
    // senders once their stores are issued; the MMA thread releases its
    // remote arrives.
    if (warp == 1) ptx::cluster_arrive_release();
    else ptx::cluster_arrive_relaxed();
    ptx::cluster_wait();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
    clock_record_end(p);
}

template <int NPAD, int OUT, bool W_MN, int RING_KB, int KIND = KIND_F16>
cudaError_t launch_gemm_splitk_cluster(const GemmParams &p, int grid, cudaStream_t stream)
{
    auto kern = gemm_splitk_cluster_kernel<NPAD, OUT, W_MN, RING_KB, KIND>;
    constexpr uint32_t smem = ClusterSplitPlan<NPAD, RING_KB>::alloc_bytes;
    static std::atomic<unsigned long long> smem_set{0};
    cudaError_t e = ensure_smem_limit(kern, smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.splits;
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

template <int NPAD, int RING_KB>
int cluster_max_splits()
{
    return ClusterSplitPlan<NPAD, RING_KB>::max_splits;
}

// stages carries the ring depth (it tells the two ring budgets apart);
// cluster = 3 marks these entries; max_active reports the largest split count
// (S-1 whole partials fit one ring).
#define TGEMM_CLUSTER_SPLIT_VARIANT_RING(NPAD, OUT, BMN, RING)                                                  \
    {NPAD, ClusterSplitPlan<NPAD, RING>::stages, OUT, BMN, ClusterSplitPlan<NPAD, RING>::alloc_bytes,          \
     &launch_gemm_splitk_cluster<NPAD, OUT, (BMN) != 0, RING>, 3, &cluster_max_splits<NPAD, RING>}
#define TGEMM_CLUSTER_SPLIT_VARIANT(NPAD, OUT, BMN) TGEMM_CLUSTER_SPLIT_VARIANT_RING(NPAD, OUT, BMN, 216), \
                                                    TGEMM_CLUSTER_SPLIT_VARIANT_RING(NPAD, OUT, BMN, 108)
// FP8 weights (B stored N x K) and activations, kind::f8f6f4
#define TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(NPAD, OUT, RING)                                                    \
    {NPAD, ClusterSplitPlan<NPAD, RING>::stages, OUT, 0, ClusterSplitPlan<NPAD, RING>::alloc_bytes,            \
     &launch_gemm_splitk_cluster<NPAD, OUT, false, RING, KIND_F8>, 3, &cluster_max_splits<NPAD, RING>, KIND_F8}
#define TGEMM_CLUSTER_SPLIT_VARIANTS_F8(OUT)                                                                     \
    TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(16, OUT, 216), TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(16, OUT, 108),        \
        TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(32, OUT, 216), TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(32, OUT, 108),    \
        TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(64, OUT, 216), TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(64, OUT, 108),    \
        TGEMM_CLUSTER_SPLIT_VARIANT_F8_RING(128, OUT, 216)

}  // namespace tgemm
