// Decoding of the tiled 4-bit weight layout into mma.m16n8k16 A fragments.
#pragma once

#include "common.cuh"

namespace flint {

// Decode one 8-row x 128-K tile pair (rows g and g+8 of a 16-row A tile) into
// A fragments of the 8 k16 steps. wg/wh: the lane's 16 code bytes of the two
// 8-row tiles; sg/sh: scale data of rows g and g+8.
template <int WFMT>
struct TileScales;

template <>
struct TileScales<0> {   // NVFP4: 8 E4M3 bytes per row (one per step)
    uint2 g, h;
};
template <>
struct TileScales<1> {   // q4_1: 4 blocks x (fp16 d, fp16 m) per row
    uint4 g, h;
};

template <int WFMT>
__device__ __forceinline__ TileScales<WFMT> load_scales(const uint8_t* base_g, const uint8_t* base_h,
                                                        int g);

template <>
__device__ __forceinline__ TileScales<0> load_scales<0>(const uint8_t* base_g, const uint8_t* base_h,
                                                        int g) {
    TileScales<0> s;
    s.g = ldg_nc_v2(base_g + g * 8);
    s.h = ldg_nc_v2(base_h + g * 8);
    return s;
}

template <>
__device__ __forceinline__ TileScales<1> load_scales<1>(const uint8_t* base_g, const uint8_t* base_h,
                                                        int g) {
    TileScales<1> s;
    s.g = ldg_nc_v4(base_g + g * 16);
    s.h = ldg_nc_v4(base_h + g * 16);
    return s;
}

// The same scales read from shared memory (a staged copy of the tile layout).
template <int WFMT>
__device__ __forceinline__ TileScales<WFMT> lds_scales(const uint8_t* base_g, const uint8_t* base_h, int g) {
    TileScales<WFMT> s;
    if constexpr (WFMT == 0) {
        s.g = *reinterpret_cast<const uint2*>(base_g + g * 8);
        s.h = *reinterpret_cast<const uint2*>(base_h + g * 8);
    } else {
        s.g = *reinterpret_cast<const uint4*>(base_g + g * 16);
        s.h = *reinterpret_cast<const uint4*>(base_h + g * 16);
    }
    return s;
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ uint32_t u2_get(const uint2& v, int i) { return i == 0 ? v.x : v.y; }

// q4_1 block parameters: one 32-bit word holds fp16 d (low half) and fp16 m
// (high half); both convert to fp32 exactly.
__device__ __forceinline__ float2 q41_dm(uint32_t word) {
    return __half22float2(*reinterpret_cast<const __half2*>(&word));
}

// q4_1 weight value, fp32(d*q + m) rounded once (d*q is exact in fp32). This
// is what the dequantisation export returns; the forward never forms it (see
// mma_k128<1>).
__device__ __forceinline__ float q41_weight(uint32_t code_byte, int high_nibble, uint32_t dm_word) {
    const uint32_t q2 = q4x2_to_f16x2(code_byte);
    const __half2 qh = *reinterpret_cast<const __half2*>(&q2);
    const float q = high_nibble ? __high2float(qh) : __low2float(qh);
    const float2 dm = q41_dm(dm_word);
    return fmaf(dm.x, q, dm.y);
}

// NVFP4 weight before its fp32 tensor scale: E2M1(code) * E4M3(scale) in fp16,
// which is exact (2 x 4 significant bits, magnitudes 2^-10 .. 2688).
__device__ __forceinline__ float nvfp4_code_times_scale(uint32_t code_byte, int high_nibble, uint32_t scale_byte) {
    uint32_t f0, f1, f2, f3;
    e2m1x8_to_f16x2(code_byte, f0, f1, f2, f3);
    const uint32_t p = hmul2_u(f0, bcast_lo(e4m3x2_to_f16x2(scale_byte)));
    const __half2 ph = *reinterpret_cast<const __half2*>(&p);
    return high_nibble ? __high2float(ph) : __low2float(ph);
}

// a[s][0..3] = A fragment registers of step s.
// NVFP4: the fp16 products E2M1 x E4M3 (exact); the tensor scale is applied
// to the fp32 accumulator by the caller.
// q4_1: the codes q themselves (integers 0..15, exact in fp16); d and m are
// applied per 32-element block by mma_k128<1>, so no weight is rounded.
template <int WFMT>
__device__ __forceinline__ void decode_tile(const uint4& wg, const uint4& wh, const TileScales<WFMT>& sc,
                                            uint32_t (&a)[8][4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // word j holds steps 2j, 2j+1
        const uint32_t xg = u4_get(wg, j), xh = u4_get(wh, j);
        if constexpr (WFMT == 0) {
            uint32_t g0, g1, g2, g3, h0, h1, h2, h3;
            e2m1x8_to_f16x2(xg, g0, g1, g2, g3);
            e2m1x8_to_f16x2(xh, h0, h1, h2, h3);
            // scale bytes of steps 2j, 2j+1: bytes 2j, 2j+1 of the row's 8 bytes
            const uint32_t sgw = u2_get(sc.g, j >> 1) >> ((j & 1) * 16);
            const uint32_t shw = u2_get(sc.h, j >> 1) >> ((j & 1) * 16);
            const uint32_t sg2 = e4m3x2_to_f16x2(sgw), sh2 = e4m3x2_to_f16x2(shw);
            const uint32_t sg_a = bcast_lo(sg2), sg_b = bcast_hi(sg2);
            const uint32_t sh_a = bcast_lo(sh2), sh_b = bcast_hi(sh2);
            a[2 * j][0] = hmul2_u(g0, sg_a);
            a[2 * j][1] = hmul2_u(h0, sh_a);
            a[2 * j][2] = hmul2_u(g1, sg_a);
            a[2 * j][3] = hmul2_u(h1, sh_a);
            a[2 * j + 1][0] = hmul2_u(g2, sg_b);
            a[2 * j + 1][1] = hmul2_u(h2, sh_b);
            a[2 * j + 1][2] = hmul2_u(g3, sg_b);
            a[2 * j + 1][3] = hmul2_u(h3, sh_b);
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int s = 2 * j + (b >> 1);
                const int lo = (b & 1) * 2;   // byte 0/2 -> k 2c.., byte 1/3 -> k 2c+8..
                a[s][lo + 0] = q4x2_to_f16x2((xg >> (8 * b)) & 0xffu);
                a[s][lo + 1] = q4x2_to_f16x2((xh >> (8 * b)) & 0xffu);
            }
        }
    }
}

// Sums of the B operand over each 32-element block of a 128-K tile, for the
// fragment columns of this lane: sx[j][0] = sum over block j of column 2c,
// sx[j][1] of column 2c+1 (c = lane % 4). Computed by the tensor core with an
// all-ones A operand, so they are sums of exactly the fp16 values the weight
// products use, accumulated in fp32. Needed by q4_1 only.
__device__ __forceinline__ void block_sums_q41(const uint32_t (&b)[16], float (&sx)[4][2]) {
    constexpr uint32_t kOnes = 0x3C003C00u;   // fp16 1.0 pair
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float t[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(t, kOnes, kOnes, kOnes, kOnes, b[4 * j], b[4 * j + 1]);
        mma_16816(t, kOnes, kOnes, kOnes, kOnes, b[4 * j + 2], b[4 * j + 3]);
        sx[j][0] = t[0];
        sx[j][1] = t[1];
    }
}

// acc (an m16n8 C fragment: rows g, g+8, columns 2c, 2c+1) += W_tile . B over
// one 128-K tile, fa from decode_tile<WFMT>, b the B fragments of the 8 steps.
// NVFP4: one mma chain. q4_1: per 32-element block j the chain of its two
// steps gives S = sum q*x exactly up to fp32 accumulation, and
//   acc += d_j * S + m_j * sum x,
// which is sum (d_j*q + m_j) * x regrouped: the weights d*q + m enter with no
// rounding of their own. sx comes from block_sums_q41 (unused for NVFP4).
template <int WFMT>
__device__ __forceinline__ void mma_k128(float (&acc)[4], const uint32_t (&fa)[8][4], const uint32_t (&b)[16],
                                         const TileScales<WFMT>& sc, const float (&sx)[4][2]) {
    if constexpr (WFMT == 0) {
#pragma unroll
        for (int s = 0; s < 8; ++s) mma_16816(acc, fa[s][0], fa[s][1], fa[s][2], fa[s][3], b[2 * s], b[2 * s + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float t[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(t, fa[2 * j][0], fa[2 * j][1], fa[2 * j][2], fa[2 * j][3], b[4 * j], b[4 * j + 1]);
            mma_16816(t, fa[2 * j + 1][0], fa[2 * j + 1][1], fa[2 * j + 1][2], fa[2 * j + 1][3], b[4 * j + 2],
                      b[4 * j + 3]);
            const float2 dg = q41_dm(u4_get(sc.g, j)), dh = q41_dm(u4_get(sc.h, j));
            acc[0] = fmaf(dg.x, t[0], fmaf(dg.y, sx[j][0], acc[0]));
            acc[1] = fmaf(dg.x, t[1], fmaf(dg.y, sx[j][1], acc[1]));
            acc[2] = fmaf(dh.x, t[2], fmaf(dh.y, sx[j][0], acc[2]));
            acc[3] = fmaf(dh.x, t[3], fmaf(dh.y, sx[j][1], acc[3]));
        }
    }
}

}  // namespace flint
