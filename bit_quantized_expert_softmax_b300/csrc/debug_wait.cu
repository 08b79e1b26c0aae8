// Bounded waits that run out on purpose: the check that a kernel whose wait
// gives up records FLINT_ETIMEOUT in the status word and returns, leaving the
// context and the handle usable. Nothing here can hang: each wait has an
// iteration limit the caller passes, and no copy or MMA is in flight while it
// waits.
#include "kernels.cuh"
#include "umma.cuh"

namespace flint {

namespace {

// kind 0: an mbarrier that expects two arrivals and gets one, so its phase
// never completes; one thread polls it `limit` times.
__global__ void mbar_timeout_kernel(uint32_t limit, uint32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 2);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive(&bar);
        mbar_wait_limit(&bar, 0, status, limit);
    }
}

// kind 1: a grid barrier of a cooperative launch of two CTAs in which CTA 1
// never arrives; CTA 0 arrives and waits `limit` polls. The counter is the
// caller's own (zeroed before the launch), never the layer's barrier counter.
__global__ void grid_timeout_kernel(unsigned long long* count, uint32_t limit, uint32_t* status) {
    GridSync gs = grid_sync_init(count, gridDim.x);
    if (blockIdx.x != 0) return;
    grid_arrive(gs);
    grid_wait(gs, status, limit);
}

}  // namespace

cudaError_t launch_wait_timeout(int kind, uint32_t limit, unsigned long long* count, uint32_t* status,
                                cudaStream_t st) {
    if (kind == 0) {
        mbar_timeout_kernel<<<1, 32, 0, st>>>(limit, status);
        return cudaGetLastError();
    }
    cudaError_t e = cudaMemsetAsync(count, 0, sizeof(unsigned long long), st);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grid_timeout_kernel, count, limit, status);
}

}  // namespace flint
