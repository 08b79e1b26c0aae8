// Token -> expert bucketing that allocates nothing.
//
// flint_moe_bucket runs on a handle, and creating a handle allocates the
// per-token workspace with cudaMalloc. Some callers cannot allocate at the
// point where they need this step: a process whose device memory is already
// reserved by another allocator (a framework's caching pool holds nearly all
// of it, so a raw cudaMalloc fails or forces that pool to release memory), a
// plugin whose host runtime forbids allocations outside its own allocator, or
// a latency-critical loop that cannot afford cudaMalloc's implicit device
// synchronisation. This file gives them the same bucketing with its scratch in
// one fixed static device array instead of a workspace.
//
// The scratch holds, per chunk of 2048 assignments, one first-output-position
// per expert: at most 256 chunks x 256 experts x 4 B = 256 KiB. Every GPU that
// loads the library holds that array until the process exits. Each call
// overwrites every scratch entry it reads before reading it, so nothing
// carries over from the previous call; but all calls on one device share the
// array, so two calls that overlap on the GPU (different streams, or host
// threads racing) corrupt each other's results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/flint_moe.h"
#include "common.cuh"

namespace {

constexpr int kNaThreads = 256;
constexpr int kNaChunk = 2048;                           // assignments per CTA
constexpr int kNaMaxAssign = 1 << 19;                    // T*k limit (65536 tokens x 8)
constexpr int kNaMaxChunks = kNaMaxAssign / kNaChunk;    // 256
constexpr int kNaMaxExperts = 256;
constexpr int kNaMaxDevices = 64;

static __device__ __align__(256) int g_bucket_scratch[kNaMaxChunks * kNaMaxExperts];

// Device address of g_bucket_scratch, looked up once per device and context:
// a cudaDeviceReset gives the device a new primary context in which the
// module, and with it the array, may sit at another address, so the address
// is looked up again when the current context is not the one it was found in.
void* g_scratch_addr[kNaMaxDevices];
CUcontext g_scratch_ctx[kNaMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// Per-expert counts of one chunk, written for every expert.
__global__ void __launch_bounds__(kNaThreads) na_hist(const int* __restrict__ sel, int n, int E,
                                                      int* __restrict__ scratch) {
    __shared__ int cnt[kNaMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int a0 = blockIdx.x * kNaChunk, a1 = min(n, a0 + kNaChunk);
    for (int a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
        const int e = sel[a];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) scratch[blockIdx.x * E + e] = cnt[e];
}

// Exclusive offsets over experts, and each chunk's first output position per
// expert (in place over the counts).
__global__ void __launch_bounds__(kNaThreads) na_scan(int n_chunks, int E, int* __restrict__ scratch,
                                                      int* __restrict__ offsets) {
    __shared__ int tot[kNaMaxExperts];
    __shared__ int off[kNaMaxExperts + 1];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int s = 0;
#pragma unroll 8
        for (int c = 0; c < n_chunks; ++c) s += scratch[c * E + e];
        tot[e] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            off[e] = run;
            run += tot[e];
        }
        off[E] = run;
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = off[e];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = off[e];
#pragma unroll 8
        for (int c = 0; c < n_chunks; ++c) {
            const int h = scratch[c * E + e];
            scratch[c * E + e] = run;
            run += h;
        }
    }
}

// Stable placement of one chunk: rounds of 256 assignments, ranks from warp
// match plus per-warp counts, so equal experts keep their assignment order.
__global__ void __launch_bounds__(kNaThreads) na_place(const int* __restrict__ sel, int n, int E,
                                                       const int* __restrict__ scratch,
                                                       int* __restrict__ perm) {
    __shared__ int base[kNaMaxExperts];
    __shared__ int wcnt[8 * kNaMaxExperts];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = scratch[blockIdx.x * E + e];
    const int a0 = blockIdx.x * kNaChunk, a1 = min(n, a0 + kNaChunk);
    for (int r0 = a0; r0 < a1; r0 += kNaThreads) {
        for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
        __syncthreads();
        const int a = r0 + threadIdx.x;
        int e = -1;
        if (a < a1) {
            e = sel[a];
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(m & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(m);
        __syncthreads();
        for (int x = threadIdx.x; x < E; x += blockDim.x) {
            int run = base[x];
            for (int w = 0; w < 8; ++w) {
                const int c = wcnt[w * E + x];
                wcnt[w * E + x] = run;
                run += c;
            }
            base[x] = run;
        }
        __syncthreads();
        if (e >= 0) perm[wcnt[warp * E + e] + rank] = a;
        __syncthreads();
    }
}

}  // namespace

extern "C" flint_status flint_moe_bucket_noalloc(const int32_t* idx_dev, int T, int k, int E,
                                                 int32_t* offsets_dev, int32_t* perm_dev, void* stream) {
    if (T < 0 || k < 1 || k > 8 || E < 1 || E > kNaMaxExperts) return FLINT_EINVAL;
    if ((long long)T * k > kNaMaxAssign) return FLINT_EINVAL;   // beyond the static scratch
    if (T == 0) return FLINT_OK;
    if (idx_dev == nullptr || offsets_dev == nullptr || perm_dev == nullptr) return FLINT_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_ECUDA;
    if (dev < 0 || dev >= kNaMaxDevices) return FLINT_ENOTIMPL;
    void* scratch = nullptr;
    {
        // the first call on a device (and the first after its context was
        // reset) finds the array's device address; later calls reuse it
        CtxGetCurrentFn get_ctx = ctx_get_current();
        if (get_ctx == nullptr) return FLINT_ECUDA;
        CUcontext ctx = nullptr;   // stays null if no context is current yet
        if (get_ctx(&ctx) != CUDA_SUCCESS) return FLINT_ECUDA;
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (ctx == nullptr || g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
            void* p = nullptr;   // the lookup makes the device's primary context current
            if (cudaGetSymbolAddress(&p, g_bucket_scratch) != cudaSuccess || p == nullptr) return FLINT_ECUDA;
            if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return FLINT_ECUDA;
            g_scratch_addr[dev] = p;
            g_scratch_ctx[dev] = ctx;
        }
        scratch = g_scratch_addr[dev];
    }
    const int n = T * k;
    const int n_chunks = (n + kNaChunk - 1) / kNaChunk;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* s = static_cast<int*>(scratch);
    na_hist<<<n_chunks, kNaThreads, 0, st>>>(idx_dev, n, E, s);
    na_scan<<<1, kNaThreads, 0, st>>>(n_chunks, E, s, offsets_dev);
    na_place<<<n_chunks, kNaThreads, 0, st>>>(idx_dev, n, E, s, perm_dev);
    return cudaGetLastError() == cudaSuccess ? FLINT_OK : FLINT_ECUDA;
}
