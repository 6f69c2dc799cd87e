// Diagnostic kernels.
//
// Self-test of the bounded-wait routine: one block waits on an mbarrier that
// nothing ever signals.  The wait must give up after `timeout_ns`, record a
// timeout fault code in the status word and let the kernel return normally.
//
// Tile-order probe: every tile number of a grid mapped on the device by the
// same grouped_tile32 the GEMM kernels use, so that tests can compare the
// device's order with the host's.
#include "tgemm_params.h"
#include "tgemm_ptx.cuh"
#include "tgemm_sched.h"
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

__global__ void tile_order_probe_kernel(int32_t tiles_m, int32_t tiles_n, int32_t group_m, int32_t count,
                                        int32_t *rows, int32_t *cols)
{
    for (int32_t bid = (int32_t)(blockIdx.x * blockDim.x + threadIdx.x); bid < count;
         bid += (int32_t)(gridDim.x * blockDim.x)) {
        int32_t r, c;
        grouped_tile32(tiles_m, tiles_n, group_m, bid, r, c);
        rows[bid] = r;
        cols[bid] = c;
    }
}

cudaError_t launch_tile_order_probe(int32_t tiles_m, int32_t tiles_n, int32_t group_m, int32_t count, int32_t *rows,
                                    int32_t *cols, cudaStream_t st)
{
    const int threads = 256;
    int blocks = (int)((count + threads - 1) / threads);
    if (blocks > 1024) blocks = 1024;
    tile_order_probe_kernel<<<blocks, threads, 0, st>>>(tiles_m, tiles_n, group_m, count, rows, cols);
    return cudaGetLastError();
}

}  // namespace tgemm
