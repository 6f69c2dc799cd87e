// Bounded pipeline waits.
//
// Every mbarrier wait in the kernels goes through wait_bounded(): it spins on
// mbarrier.try_wait (which itself suspends the thread for a short, hardware
// chosen time) and, every 64 polls, checks the CTA's abort flag and the
// elapsed %globaltimer time.  On expiry it records a fault code in the device
// status word (the first fault wins), raises the abort flag so that the
// other roles stop waiting too, and returns false.  No trap and no assert:
// the kernel winds down and the context stays usable.  This answers the
// "silent deadlock" risk of hand-written warp-specialised pipelines that the
// Croqtile tutorial ("How to optimise a matrix-multiply kernel step by step
// with Croqtile") names in its summary.
#pragma once

#include "tgemm_params.h"
#include "tgemm_ptx.cuh"

namespace tgemm {

struct WaitCtx {
    uint32_t *status;            // device status word
    volatile int *abort_flag;    // in shared memory, one per CTA
    uint64_t timeout_ns;
    uint32_t peer_abort = 0;     // shared::cluster address of the pair partner's flag (0: none)
    uint32_t peer_mask = 0;      // or: cluster ranks whose flag (at abort_local) is raised too
    uint32_t abort_local = 0;    // shared::cta address of the flag, for peer_mask
};

__device__ __forceinline__ void record_fault(const WaitCtx &w, uint32_t site)
{
    const uint32_t code = (kFaultTimeout << 28) | ((site & 0xffu) << 20) | (blockIdx.x & 0xfffffu);
    *w.abort_flag = 1;
    if (w.peer_abort)   // the partner CTA of a pair winds down too
        asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(w.peer_abort), "r"(1) : "memory");
    for (uint32_t r = 0; r < 8; ++r)   // every CTA of a larger cluster that shares this one's copies
        if ((w.peer_mask >> r) & 1u) {
            const uint32_t a = ptx::map_to_cta(w.abort_local, r);
            asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(1) : "memory");
        }
    if (w.status) atomicCAS(w.status, 0u, code);
}

// honour_abort = false is used by the wind-down waits (in-flight copies and
// MMAs) that must still be waited for after the abort flag went up.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, WaitCtx w, uint32_t site,
                                              bool honour_abort)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t poll = 1;; ++poll) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((poll & 63u) == 0) {
            if (honour_abort && *w.abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
                record_fault(w, site);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx &w,
                                             uint32_t site, bool honour_abort = true)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, w, site, honour_abort);
}

}  // namespace tgemm
