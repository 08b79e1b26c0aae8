// Dense block-scaled FP4 tensor-core throughput of this GPU, measured: every
// SM issues back-to-back tcgen05.mma kind::mxf4nvf4 (scale_vec::4X, M = 128,
// N = 128 or 256, K = 64, fp32 accumulation) on operands resident in shared
// memory and scale factors resident in tensor memory, so nothing but the
// tensor pipe is timed. The result is the denominator of the FP4 roofline
// fractions the benchmark reports.
#include "kernels.cuh"
#include "umma.cuh"

namespace flint {

namespace {

constexpr int kPThreads = 128;
constexpr int kPABytes = 128 * 128;            // A: 128 rows x 256 E2M1, 128-byte swizzled rows
constexpr int kPSmem = 120 * 1024;             // more than half an SM's shared memory: one CTA per SM

template <int N>
__global__ void __launch_bounds__(kPThreads, 1) fp4_peak_kernel(int iters, uint32_t* status) {
    extern __shared__ uint8_t praw[];
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tmem_base;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(praw) + 1023) & ~uintptr_t(1023));
    constexpr int kBBytes = N * 128;
    static_assert(kPABytes + kBBytes + 1024 <= kPSmem, "operands fit");
    const int warp = threadIdx.x >> 5;
    // operands: E2M1 code 2 (value 1.0) in every nibble
    for (int i = threadIdx.x * 16; i < kPABytes + kBBytes; i += kPThreads * 16)
        *reinterpret_cast<uint4*>(sm + i) = make_uint4(0x22222222u, 0x22222222u, 0x22222222u, 0x22222222u);
    fence_proxy_async_smem();   // the generic-proxy writes are seen by the tensor core
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // scale factors UE4M3 1.0 (0x38) in columns 256..319 of every lane; the
    // MMAs read A's at 256 + 4j and B's at 288 + 8j
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int c = 0; c < 64; c += 4) tmem_st4(tmem + lane_base + 256 + c, 0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        const uint32_t idesc = idesc_nvfp4_f32(128, N);
        const uint64_t da = sdesc_kmajor_sw128(sm), db = sdesc_kmajor_sw128(sm + kPABytes);
#pragma unroll 1
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                umma_nvfp4(tmem, da + 2 * j, db + 2 * j, idesc, tmem + 256 + 4 * j, tmem + 288 + 8 * j, (it | j) != 0);
        }
        umma_commit(&done);
        bool got = false;
        for (uint32_t k = 0; k < (1u << 24) && !got; ++k) {   // at most a few seconds
            got = mbar_try_wait(&done, 0);
            if (!got) __nanosleep(256);
        }
        if (!got) atomicOr(status, kStatusTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_fp4_peak(int n, int iters, int n_sms, uint32_t* status, cudaStream_t st) {
    void (*kern)(int, uint32_t*) = n == 256 ? fp4_peak_kernel<256> : fp4_peak_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
    if (e != cudaSuccess) return e;
    kern<<<n_sms, kPThreads, kPSmem, st>>>(iters, status);
    return cudaGetLastError();
}

}  // namespace flint
