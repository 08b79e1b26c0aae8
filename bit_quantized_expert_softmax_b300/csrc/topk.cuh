// Top-k selection with renormalised softmax weights, one warp per token.
#pragma once

#include "common.cuh"

namespace flint {

// ---------------------------------------------------------------------------
// a2: top-k of one token's logits by one warp
// ---------------------------------------------------------------------------
// kCG: read the logits with ld.global.cg (global memory written by other CTAs
// of the same kernel); otherwise a generic load (shared or global memory).
template <bool kCG>
__device__ __forceinline__ void topk_warp(const float* __restrict__ Lrow, int E, int k, int* __restrict__ idx_out,
                          float* __restrict__ w_out, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const int n = E >> 5;
    float v[8];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < n) {
            float x = kCG ? __ldcg(Lrow + i * 32 + lane) : Lrow[i * 32 + lane];
            if (!isfinite(x)) {
                bad = true;
                x = -INFINITY;
            }
            v[i] = x;
        } else {
            v[i] = -INFINITY;
        }
    }
    if (status != nullptr && __any_sync(0xffffffffu, bad) && lane == 0)
        atomicOr(status, kStatusNonFiniteLogit);
    uint32_t taken = 0;
    float sel_v[8];
    int sel_i[8];
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < n && !((taken >> i) & 1u)) {
                int e = i * 32 + lane;
                if (v[i] > bv || (v[i] == bv && e < bi)) {
                    bv = v[i];
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        sel_v[j] = bv;
        sel_i[j] = bi;
    }
    // renormalised softmax over the selected logits (sel_v[0] is the maximum)
    float sum = 0.f;
    float ex[8];
    for (int j = 0; j < k; ++j) {
        ex[j] = expf(sel_v[j] - sel_v[0]);
        sum += ex[j];
    }
    if (lane < k) {
        float e = 0.f;
        int id = 0;
        for (int j = 0; j < k; ++j)
            if (j == lane) {
                e = ex[j];
                id = sel_i[j];
            }
        idx_out[lane] = id;
        if (w_out != nullptr) w_out[lane] = e / sum;
    }
}

}  // namespace flint
