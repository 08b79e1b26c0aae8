// Top-k selection with renormalised softmax weights, one warp per token.
#pragma once

#include "common.cuh"

namespace flint {

// ---------------------------------------------------------------------------
// a2: top-k of one token's logits by one warp
// ---------------------------------------------------------------------------
// kCG: read the logits with ld.global.cg (global memory written by other CTAs
// of the same kernel); otherwise a generic load (shared or global memory).
// Returns, in lane j < k, the expert of selection j (-1 in the other lanes).
template <bool kCG>
__device__ __forceinline__ int topk_warp(const float* __restrict__ Lrow, int E, int k, int* __restrict__ idx_out,
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
    float my_v = 0.f;   // lane j < k ends with selection j
    int my_i = 0;
    // one selection per round; the round is not unrolled (the code runs once
    // per token and its size, not its trip count, sets its cost)
#pragma unroll 1
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
        const int wi =
            (int)__reduce_min_sync(0xffffffffu, (bk == mk && bi != 0x7fffffff) ? (uint32_t)bi : 0xffffffffu);
        if ((wi & 31) == lane) taken |= 1u << (wi >> 5);
        if (lane == j) {
            my_v = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk);
            my_i = wi;
        }
    }
    // renormalised softmax over the selected logits (selection 0 is the maximum)
    const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < k ? expf(my_v - v0) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
        idx_out[lane] = my_i;
        if (w_out != nullptr) w_out[lane] = ex / sum;
    }
    return lane < k ? my_i : -1;
}

}  // namespace flint
