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
    // Order-preserving unsigned key of a float (-0.0 folded onto +0.0 so that
    // equal values compare equal); the warp max of keys picks the value, the
    // warp min of indices among lanes holding it picks the lower expert.
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = __float_as_uint(v[i] + 0.0f);
        key[i] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    }
    uint32_t taken = 0;
    float sel_v[8];
    int sel_i[8];
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0u;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < n && !((taken >> i) & 1u) && (key[i] > bk || bi == 0x7fffffff)) {
                bk = key[i];
                bi = i * 32 + lane;
            }
        }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const int wi = (int)__reduce_min_sync(0xffffffffu, (bk == mk && bi != 0x7fffffff) ? (uint32_t)bi : 0xffffffffu);
        if ((wi & 31) == lane) taken |= 1u << (wi >> 5);
        const uint32_t wb = (mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk;
        sel_v[j] = __uint_as_float(wb);
        sel_i[j] = wi;
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
