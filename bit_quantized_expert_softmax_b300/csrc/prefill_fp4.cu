// Large-T (prefill) kernels on the 5th-generation tensor cores.
//
// Router logits for many tokens: L = x . W_r^T + b is a dense contraction
// (T x d) x (d x E). The hidden states are bf16 and therefore exact in bf16;
// the fp32 router is split once at load time into two bf16 matrices,
// W_r = W_hi + W_lo (W_hi = bf16(W_r), W_lo = bf16(W_r - W_hi)), whose sum
// keeps about 16 significant bits. Two bf16 x bf16 tensor-core products with
// fp32 accumulation then give the logits within ~2^-16 relative of the fp32
// reference, well inside the router's 1e-4 tolerance, at tensor-core speed.
//
// Kernel structure (one CTA per 128 x 128 output tile, 192 threads):
//   warp 0      TMA producer: x, W_hi, W_lo tiles of 64 K-elements into a
//               4-stage shared-memory ring (128-byte swizzle)
//   warp 1      allocates 128 TMEM columns; one thread issues the MMAs
//               (M=128, N=128, K=16 each) and commits each stage back
//   warps 2..5  epilogue: TMEM -> registers (+ bias) -> global fp32
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "pdl.cuh"
#include "umma.cuh"

namespace flint {

namespace {

constexpr int kRM = 128, kRN = 128, kRK = 64, kRStages = 4;
constexpr int kRTileBytes = kRM * kRK * 2;                 // 16 KiB per operand tile
constexpr int kRStageBytes = 3 * kRTileBytes;              // x, W_hi, W_lo
constexpr int kRSmem = kRStages * kRStageBytes + 1024;     // + alignment slack
constexpr int kRThreads = 192;

struct RouterUmmaArgs {
    float* logits;
    const float* bias;
    int T, E, nkb;
    uint32_t* status;
};

__global__ void __launch_bounds__(kRThreads, 1)
    router_umma_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mwh,
                       const __grid_constant__ CUtensorMap mwl, RouterUmmaArgs a) {
    griddep_wait();
    extern __shared__ uint8_t rsm_raw[];
    __shared__ __align__(8) uint64_t full[kRStages], empty[kRStages], done;
    __shared__ uint32_t tmem_base;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rsm_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kRM, n0 = blockIdx.y * kRN;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0 && lane == 0) {
        // producer
        uint32_t fills = 0;
        for (int kb = 0; kb < a.nkb; ++kb) {
            const int s = kb % kRStages;
            if (kb >= kRStages && !mbar_wait_bounded(&empty[s], (uint32_t)((kb / kRStages - 1) & 1), a.status))
                break;
            uint8_t* st = sm + s * kRStageBytes;
            mbar_arrive_expect_tx(&full[s], kRStageBytes);
            tma_load_2d(st, &mx, kb * kRK, m0, &full[s]);
            tma_load_2d(st + kRTileBytes, &mwh, kb * kRK, n0, &full[s]);
            tma_load_2d(st + 2 * kRTileBytes, &mwl, kb * kRK, n0, &full[s]);
            ++fills;
        }
        drain_ring(full, kRStages, fills, a.status);   // no copy still in flight at exit
    } else if (warp == 1 && lane == 0) {
        // MMA issue
        const uint32_t idesc = idesc_bf16_f32(kRM, kRN);
        bool ok = true;
        for (int kb = 0; kb < a.nkb && ok; ++kb) {
            const int s = kb % kRStages;
            ok = mbar_wait_bounded(&full[s], (uint32_t)((kb / kRStages) & 1), a.status);
            if (!ok) break;
            tc_fence_after();
            const uint8_t* st = sm + s * kRStageBytes;
            const uint64_t da = sdesc_kmajor_sw128(st);
            const uint64_t dh = sdesc_kmajor_sw128(st + kRTileBytes);
            const uint64_t dl = sdesc_kmajor_sw128(st + 2 * kRTileBytes);
#pragma unroll
            for (int k = 0; k < kRK / 16; ++k)   // 16 bf16 = 32 bytes = 2 descriptor units per step
                umma_bf16(tmem, da + 2 * k, dh + 2 * k, idesc, (kb | k) != 0);
#pragma unroll
            for (int k = 0; k < kRK / 16; ++k) umma_bf16(tmem, da + 2 * k, dl + 2 * k, idesc, 1u);
            umma_commit(&empty[s]);
        }
        umma_commit(&done);
        mbar_wait_bounded(&done, 0, a.status);   // no MMA still running when the TMEM is released
    } else if (warp >= 2) {
        // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (rows of the tile)
        const int quad = warp & 3;
        const bool ok = mbar_wait_bounded(&done, 0, a.status);
        tc_fence_after();
        const int row = m0 + quad * 32 + lane;
        if (ok) {
#pragma unroll 1
            for (int c = 0; c < kRN / 16; ++c) {
                uint32_t r[16];
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c * 16, r);
                tmem_ld_wait();
                if (row < a.T) {
                    float* dst = a.logits + (size_t)row * a.E + n0 + c * 16;
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        float4 v;
                        v.x = __uint_as_float(r[i + 0]) + __ldg(a.bias + n0 + c * 16 + i + 0);
                        v.y = __uint_as_float(r[i + 1]) + __ldg(a.bias + n0 + c * 16 + i + 1);
                        v.z = __uint_as_float(r[i + 2]) + __ldg(a.bias + n0 + c * 16 + i + 2);
                        v.w = __uint_as_float(r[i + 3]) + __ldg(a.bias + n0 + c * 16 + i + 3);
                        *reinterpret_cast<float4*>(dst + i) = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// W_hi = bf16(W), W_lo = bf16(W - W_hi), both round-to-nearest-even.
__global__ void split_router_kernel(const float* __restrict__ w, __nv_bfloat16* __restrict__ hi,
                                    __nv_bfloat16* __restrict__ lo, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = w[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        hi[i] = h;
        lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

}  // namespace

// 2-D tensor map of a row-major bf16 matrix [rows x cols], boxes of 128 rows x
// 64 columns with the 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rows, int cols) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t prepare_prefill() {
    cudaError_t e = cudaFuncSetAttribute(router_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

cudaError_t split_router(const float* w, __nv_bfloat16* hi, __nv_bfloat16* lo, size_t n, cudaStream_t st) {
    split_router_kernel<<<148 * 4, 256, 0, st>>>(w, hi, lo, n);
    return cudaGetLastError();
}

bool router_umma_supported(const Shape& s) { return s.E % kRN == 0 && s.d % kRK == 0 && encode_fn() != nullptr; }

cudaError_t launch_router_umma(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T, float* logits,
                               uint32_t* status, cudaStream_t st) {
    CUtensorMap mx;
    if (!make_tmap_bf16(&mx, x, T, s.d)) return cudaErrorInvalidValue;
    RouterUmmaArgs a{logits, L.bias, T, s.E, s.d / kRK, status};
    dim3 grid((T + kRM - 1) / kRM, s.E / kRN);
    return launch_pdl(router_umma_kernel, grid, dim3(kRThreads), kRSmem, st, mx, L.tmap_router_hi, L.tmap_router_lo, a);
}

}  // namespace flint
