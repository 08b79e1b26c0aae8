// Packing of NVFP4 matrices into swizzled tiles and the single-matrix
// block-scaled FP4 GEMM entry point built on fp4_gemm_kernel.
#include "../../include/flint_moe.h"
#include "gemm_fp4.cuh"
#include "kernels.cuh"

namespace flint {

namespace {

// Canonical row-major NVFP4 (codes [R][K/2], E4M3 scales [R][K/16]) ->
// blocks: block (rt, kt) of 128 rows x 256 elements at blocks + (rt*KT + kt) *
// 18 KiB, its swizzled codes first and its scales after them.
// One thread per 16 bytes of codes.
__global__ void pack_fp4_tiles_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                      uint8_t* __restrict__ blocks, int R, int K) {
    const int KT = K / kGK;
    const long n16 = (long)R * (K / 2) / 16;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n16; i += (long)gridDim.x * blockDim.x) {
        const long byte = i * 16;
        const int row = (int)(byte / (K / 2));
        const int col = (int)(byte % (K / 2));      // byte within the row
        const int rt = row / kGM, r = row % kGM;
        const int kt = col / 128, j = col % 128;    // 128 bytes (256 elements) per k-tile
        uint8_t* blk = blocks + ((size_t)rt * KT + kt) * kGBlk;
        const uint4 v = *reinterpret_cast<const uint4*>(codes + byte);
        *reinterpret_cast<uint4*>(blk + swz_offset(r, j)) = v;
        // scales: this 16-byte chunk covers 32 elements = 2 scale bytes
        const uint8_t* s = scales + (size_t)row * (K / 16) + col / 8;
        uint8_t* d = blk + kGTile + r * 16 + j / 8;
        d[0] = s[0];
        d[1] = s[1];
    }
}

struct DebugGemm {
    const uint8_t* a;
    const uint8_t* b;
    float* d;
    int mt, nt, kt, N;
    __device__ int n_items() const { return mt * nt; }
    struct Pre {};
    __device__ Pre pre(const Fp4Item&, int, int) const { return {}; }
    __device__ void item(int i, Fp4Item& w) const {
        const int m = i / nt, n = i % nt;
        w.a = a + (size_t)m * kt * kGBlk;
        w.b = b + (size_t)n * kt * kGBlk;
        w.b2 = nullptr;
        w.kt = kt;
        w.m = m;
        w.n = n;
        w.aux = 0;
    }
    static constexpr int kStages = 3;
    static constexpr int kNB = 1;
    static constexpr int kKPS = 2;
    static constexpr bool kBPair = false;
    static constexpr int kEpiSmemPerWarp = 0;
    __device__ void epilogue_finish() const {}
    template <class Release>
    __device__ void epilogue(const Fp4Item& w, Pre, uint32_t taddr, int row, int half, uint8_t*,
                             Release release) const {
        float* dst = d + (size_t)(w.m * kGM + row) * N + w.n * kGN;
#pragma unroll 1
        for (int c = 4 * half; c < 4 * half + 4; ++c) {
            uint32_t r[16];
            tmem_ld16(taddr + c * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(dst + c * 16 + i) = make_float4(
                    __uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
        }
        release();
    }
};

}  // namespace

cudaError_t pack_fp4_tiles(const uint8_t* codes, const uint8_t* scales, uint8_t* blocks, int R, int K,
                           cudaStream_t st) {
    const long n16 = (long)R * (K / 2) / 16;
    long grid = (n16 + 255) / 256;
    if (grid > 148 * 16) grid = 148 * 16;
    pack_fp4_tiles_kernel<<<(int)grid, 256, 0, st>>>(codes, scales, blocks, R, K);
    return cudaGetLastError();
}

cudaError_t prepare_gemm_fp4() {
    cudaError_t e = cudaFuncSetAttribute(fp4_gemm_kernel<DebugGemm>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fp4_gemm_smem<DebugGemm>());
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

}  // namespace flint

extern "C" flint_status flint_moe_debug_fp4_gemm(const uint8_t* a_codes, const uint8_t* a_scales,
                                                 const uint8_t* b_codes, const uint8_t* b_scales, int M, int N,
                                                 int K, float* d, void* stream) {
    using namespace flint;
    if (a_codes == nullptr || a_scales == nullptr || b_codes == nullptr || b_scales == nullptr || d == nullptr)
        return FLINT_EINVAL;
    if (M <= 0 || N <= 0 || K <= 0 || M % kGM || N % kGN || K % kGK) return FLINT_EINVAL;
    if (prepare_gemm_fp4() != cudaSuccess) return FLINT_ECUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int KT = K / kGK;
    uint8_t* buf = nullptr;
    const size_t ab = (size_t)(M / kGM) * KT * kGBlk, bb = (size_t)(N / kGN) * KT * kGBlk;
    uint32_t* status = nullptr;
    if (cudaMalloc(&buf, ab + bb + 256) != cudaSuccess) return FLINT_ENOMEM;
    status = reinterpret_cast<uint32_t*>(buf + ab + bb);
    cudaError_t e = cudaMemsetAsync(status, 0, 4, st);
    if (e == cudaSuccess) e = pack_fp4_tiles(a_codes, a_scales, buf, M, K, st);
    if (e == cudaSuccess) e = pack_fp4_tiles(b_codes, b_scales, buf + ab, N, K, st);
    if (e == cudaSuccess) {
        DebugGemm p{buf, buf + ab, d, M / kGM, N / kGN, KT, N};
        const int items = (M / kGM) * (N / kGN);
        fp4_gemm_kernel<DebugGemm><<<items < 148 ? items : 148, kGThreads, fp4_gemm_smem<DebugGemm>(), st>>>(p, status);
        e = cudaGetLastError();
    }
    uint32_t hs = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&hs, status, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(buf);
    if (e != cudaSuccess) return FLINT_ECUDA;
    return hs ? FLINT_ETIMEOUT : FLINT_OK;
}
