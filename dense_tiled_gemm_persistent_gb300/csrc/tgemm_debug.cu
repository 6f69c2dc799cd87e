// Diagnostic kernels.
//
// Self-test of the bounded-wait routine: one block waits on an mbarrier that
// nothing ever signals.  The wait must give up after `timeout_ns`, record a
// timeout fault code in the status word and let the kernel return normally.
//
// Tile-order probe: every tile number of a grid mapped on the device by the
// same grouped_tile32 the GEMM kernels use, so that tests can compare the
// device's order with the host's.
//
// SM-clock probe: one thread counts %clock64 cycles over a stretch of
// %globaltimer time, which gives the SM clock of the moment the probe runs
// (for benchmark records; NVML's clock readings trail by tens of ms).
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

__global__ void sm_clock_probe_kernel(uint64_t *out, uint64_t duration_ns)
{
    if (threadIdx.x != 0) return;
    const uint64_t t0 = ptx::globaltimer_ns();
    const uint64_t c0 = clock64();
    uint64_t t = t0;
    // bounded twice: by the time asked for and by an iteration count far above it
    for (uint32_t i = 0; i < (1u << 26) && t - t0 < duration_ns; ++i) t = ptx::globaltimer_ns();
    const uint64_t c1 = clock64();
    out[0] = t - t0;
    out[1] = c1 - c0;
}

cudaError_t launch_sm_clock_probe(uint64_t *out, uint64_t duration_ns, cudaStream_t st)
{
    sm_clock_probe_kernel<<<1, 32, 0, st>>>(out, duration_ns);
    return cudaGetLastError();
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
