// Self-test of the bounded-wait routine: one block waits on an mbarrier that
// nothing ever signals.  The wait must give up after `timeout_ns`, record a
// timeout fault code in the status word and let the kernel return normally.
#include "tgemm_params.h"
#include "tgemm_ptx.cuh"
#include "tgemm_wait.cuh"

namespace tgemm {

__global__ void wait_timeout_probe_kernel(uint32_t *status, uint64_t timeout_ns)
{
    __shared__ alignas(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx w{status, &abort_flag, timeout_ns};
        wait_bounded(b, 0, w, SITE_DEBUG);   // phase 0 never completes
    }
    __syncthreads();
}

cudaError_t launch_wait_timeout_probe(uint32_t *status, uint64_t timeout_ns, cudaStream_t st)
{
    wait_timeout_probe_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace tgemm
