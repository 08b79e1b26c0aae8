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

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ uint32_t u2_get(const uint2& v, int i) { return i == 0 ? v.x : v.y; }

// a[s][0..3] = A fragment registers of step s
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
            // steps 2j, 2j+1 form 32-element block j: (d, m) word of block j
            const uint32_t dmg = u4_get(sc.g, j), dmh = u4_get(sc.h, j);
            const uint32_t dg = bcast_lo(dmg), mg = bcast_hi(dmg);
            const uint32_t dh = bcast_lo(dmh), mh = bcast_hi(dmh);
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const uint32_t qg = q4x2_to_f16x2((xg >> (8 * b)) & 0xffu);
                const uint32_t qh = q4x2_to_f16x2((xh >> (8 * b)) & 0xffu);
                const int s = 2 * j + (b >> 1);
                const int lo = (b & 1) * 2;   // byte 0/2 -> k 2c.., byte 1/3 -> k 2c+8..
                a[s][lo + 0] = hfma2_u(qg, dg, mg);
                a[s][lo + 1] = hfma2_u(qh, dh, mh);
            }
        }
    }
}

}  // namespace flint
