// Large-T (prefill) expert projections on the block-scaled FP4 tensor cores.
//
// NVFP4 weights force the FP4 x FP4 tensor-core kind, so the activations that
// enter each projection are quantised to NVFP4 as well (per row: an fp32 scale
// s = amax/2688; per 16 elements: an E4M3 scale E4M3_rne((amax_b/6)/s); codes
// E2M1_rne(v * (1/(E4M3(sb)*s)))). h enters the down projection rounded to
// bf16 first. Pipeline for one layer (after routing and bucketing):
//   plan      pad every expert's rows to a multiple of 128 (M-tile table)
//   quant_x   quantise x[token] for every padded row into swizzled A tiles
//   gemm1     gate/up: [rows x d] . [2f x d]^T, each 128-column tile holds 64
//             gate and 64 up columns of the same f range; epilogue
//             h = silu(g)*u -> bf16
//   quant_h   quantise each h row into swizzled A tiles of the down GEMM
//   gemm2     down: [rows x f] . [d x f]^T; epilogue scales by the routing
//             weight and writes (shared expert) or adds (routed) into an fp32
//             [T x d] sum
//   cast      out = bf16(sum)
#include "../../include/flint_moe.h"
#include "gemm_fp4.cuh"
#include "kernels.cuh"

namespace flint {

namespace {

// ---------------------------------------------------------------------------
// activation quantisation of one row, by one warp (lane l owns EPL
// consecutive elements)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xffu;
}

// eight floats -> four bytes of E2M1 pairs (element 2i in the low nibble of byte i)
__device__ __forceinline__ uint32_t f32x8_to_e2m1(const float* v) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t h2 = e4m3x2_to_f16x2(b & 0xffu);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

// Quantise the warp's row: v[EPL] per lane. Outputs per lane: EPL/2 code
// bytes (codes[], little-endian words) and EPL/16 scale bytes (packed into
// sbytes); returns the row scale.
template <int EPL>
__device__ __forceinline__ float quant_row(const float (&v)[EPL], uint32_t (&codes)[EPL / 8], uint32_t& sbytes) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float amax_t = warp_max(amax);
    const float s_t = amax_t / 2688.0f;
    sbytes = 0u;
#pragma unroll
    for (int b = 0; b < EPL / 16; ++b) {
        float ab = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[16 * b + i]));
        const float ratio = s_t > 0.f ? (ab / 6.0f) / s_t : 0.0f;
        const uint32_t sb = f32_to_e4m3(ratio);
        const float S = e4m3_to_f32(sb) * s_t;
        sbytes |= sb << (8 * b);
        if (S > 0.f) {
            const float inv = 1.0f / S;
            float q[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) q[i] = v[16 * b + i] * inv;
            codes[2 * b] = f32x8_to_e2m1(q);
            codes[2 * b + 1] = f32x8_to_e2m1(q + 8);
        } else {
            codes[2 * b] = 0u;
            codes[2 * b + 1] = 0u;
        }
    }
    return s_t;
}

// Write the lane's part of row r of a swizzled row tile (K elements; lane
// owns elements [lane*EPL, (lane+1)*EPL)).
template <int EPL>
__device__ __forceinline__ void store_row_swizzled(uint8_t* tiles, uint8_t* sf, int r, int lane,
                                                   const uint32_t (&codes)[EPL / 8], uint32_t sbytes) {
    const int e0 = lane * EPL;                 // first element
    const int kt = e0 / kGK;
    const int j = (e0 % kGK) / 2;              // byte within the 128-byte row of the k-tile
    uint8_t* t = tiles + (size_t)kt * kGTile;
    if constexpr (EPL >= 32) {
#pragma unroll
        for (int c = 0; c < EPL / 32; ++c)
            *reinterpret_cast<uint4*>(t + swz_offset(r, j + 16 * c)) =
                make_uint4(codes[4 * c], codes[4 * c + 1], codes[4 * c + 2], codes[4 * c + 3]);
    } else {
        *reinterpret_cast<uint2*>(t + swz_offset(r, j)) = make_uint2(codes[0], codes[1]);
    }
    uint8_t* s = sf + (size_t)kt * kGSf + r * 16 + (e0 % kGK) / 16;
    if constexpr (EPL == 64) {
        *reinterpret_cast<uint32_t*>(s) = sbytes;
    } else {
        *s = (uint8_t)sbytes;
    }
}

struct PrefillCtx {
    // routing / bucketing results
    const int* perm;
    const float* wts;
    const int* slot_expert;
    const int* slot_off;
    const int* slot_cnt;
    const int* meta;          // [0] active slots, [2] M-tiles (written by the plan kernel)
    // plan
    int* poff;                // [slots] first padded row of each slot
    int* mt_slot;             // [M-tiles]
    int* mt_m;
    // activations
    const __nv_bfloat16* x;
    uint8_t* a1;
    uint8_t* a1sf;
    float* sa;
    __nv_bfloat16* h;
    uint8_t* a2;
    uint8_t* a2sf;
    float* sh;
    float* out32;
    // weights
    const uint8_t* w1;
    const uint8_t* w1sf;
    const uint8_t* w2;
    const uint8_t* w2sf;
    const float* tscale;
    int T, d, f, E, k;
};

__device__ __forceinline__ int ctx_token(const PrefillCtx& c, int p) {
    return p < c.T * c.k ? __ldg(c.perm + p) / c.k : p - c.T * c.k;
}

// M-tile table: 128-row tiles of every active slot, padded offsets. One CTA
// of 256 threads; slot i (< 256) is handled by thread i, slot 256 (the shared
// expert when all 256 routed experts are active) by thread 0 afterwards.
__global__ void __launch_bounds__(256) plan_kernel(PrefillCtx c, int* meta_rw) {
    __shared__ int wsum[8];
    __shared__ int s_base[257];
    __shared__ int s_total;
    const int n_slots = c.meta[0];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = threadIdx.x;
    const int mt = i < n_slots ? (c.slot_cnt[i] + kGM - 1) / kGM : 0;
    int x = mt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < 8; ++w) {
            const int t = wsum[w];
            wsum[w] = run;
            run += t;
        }
        s_total = run;
    }
    __syncthreads();
    s_base[i] = wsum[warp] + x - mt;
    if (threadIdx.x == 0) {
        int run = s_total;
        for (int sl = 256; sl < n_slots; ++sl) {
            s_base[sl] = run;
            run += (c.slot_cnt[sl] + kGM - 1) / kGM;
        }
        s_total = run;
    }
    __syncthreads();
    for (int sl = threadIdx.x; sl < n_slots; sl += blockDim.x) {
        const int base = s_base[sl];
        const int m_tiles = (c.slot_cnt[sl] + kGM - 1) / kGM;
        c.poff[sl] = base * kGM;
        for (int m = 0; m < m_tiles; ++m) {
            c.mt_slot[base + m] = sl;
            c.mt_m[base + m] = m;
        }
    }
    if (threadIdx.x == 0) meta_rw[2] = s_total;
}

// Quantise x[token] of every padded row (zeros for padding rows). One warp
// per row, 8 warps per CTA, grid-stride over rows of all M-tiles.
template <int EPL>
__global__ void __launch_bounds__(256) quant_x_kernel(PrefillCtx c) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rows = c.meta[2] * kGM;
    const int KT = c.d / kGK;
    for (int row = blockIdx.x * 8 + warp; row < n_rows; row += gridDim.x * 8) {
        const int mt = row / kGM, r = row % kGM;
        const int slot = c.mt_slot[mt], m = c.mt_m[mt];
        const int q = m * kGM + r;
        const int rt = c.poff[slot] / kGM + m;
        uint8_t* tiles = c.a1 + (size_t)rt * KT * kGTile;
        uint8_t* sf = c.a1sf + (size_t)rt * KT * kGSf;
        uint32_t codes[EPL / 8];
        uint32_t sb = 0;
        float s_t = 0.f;
        if (q < c.slot_cnt[slot]) {
            const int t = ctx_token(c, c.slot_off[slot] + q);
            const __nv_bfloat16* xr = c.x + (size_t)t * c.d + lane * EPL;
            float v[EPL];
#pragma unroll
            for (int i = 0; i < EPL; i += 8) {
                const uint4 raw = *reinterpret_cast<const uint4*>(xr + i);
                const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    v[i + 2 * u] = __low2float(p2[u]);
                    v[i + 2 * u + 1] = __high2float(p2[u]);
                }
            }
            s_t = quant_row<EPL>(v, codes, sb);
        } else {
#pragma unroll
            for (int i = 0; i < EPL / 8; ++i) codes[i] = 0u;
        }
        store_row_swizzled<EPL>(tiles, sf, r, lane, codes, sb);
        if (lane == 0) c.sa[rt * kGM + r] = s_t;
    }
}

// Quantise each h row (bf16, f elements) into the down GEMM's A tiles.
template <int EPL>
__global__ void __launch_bounds__(256) quant_h_kernel(PrefillCtx c) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rows = c.meta[2] * kGM;
    const int KT = c.f / kGK;
    for (int row = blockIdx.x * 8 + warp; row < n_rows; row += gridDim.x * 8) {
        const int mt = row / kGM, r = row % kGM;
        const int slot = c.mt_slot[mt], m = c.mt_m[mt];
        const int q = m * kGM + r;
        const int rt = c.poff[slot] / kGM + m;
        uint8_t* tiles = c.a2 + (size_t)rt * KT * kGTile;
        uint8_t* sf = c.a2sf + (size_t)rt * KT * kGSf;
        uint32_t codes[EPL / 8];
        uint32_t sb = 0;
        float s_t = 0.f;
        if (q < c.slot_cnt[slot]) {
            const __nv_bfloat16* hr = c.h + (size_t)(rt * kGM + r) * c.f + lane * EPL;
            float v[EPL];
#pragma unroll
            for (int i = 0; i < EPL; i += 8) {
                const uint4 raw = *reinterpret_cast<const uint4*>(hr + i);
                const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    v[i + 2 * u] = __low2float(p2[u]);
                    v[i + 2 * u + 1] = __high2float(p2[u]);
                }
            }
            s_t = quant_row<EPL>(v, codes, sb);
        } else {
#pragma unroll
            for (int i = 0; i < EPL / 8; ++i) codes[i] = 0u;
        }
        store_row_swizzled<EPL>(tiles, sf, r, lane, codes, sb);
        if (lane == 0) c.sh[rt * kGM + r] = s_t;
    }
}

// gate/up GEMM: item = (M-tile, N-tile of 64 gate + 64 up columns)
struct Gemm1 {
    PrefillCtx c;
    int NT, KT;
    __device__ int n_items() const { return c.meta[2] * NT; }
    __device__ bool item(int i, Fp4Item& w) const {
        const int mt = i / NT, nt = i % NT;
        const int slot = c.mt_slot[mt], m = c.mt_m[mt];
        const int e = c.slot_expert[slot];
        const int rt = c.poff[slot] / kGM + m;
        w.a = c.a1 + (size_t)rt * KT * kGTile;
        w.asf = c.a1sf + (size_t)rt * KT * kGSf;
        w.b = c.w1 + ((size_t)e * NT + nt) * KT * kGTile;
        w.bsf = c.w1sf + ((size_t)e * NT + nt) * KT * kGSf;
        w.kt = KT;
        w.m = m;
        w.n = nt;
        w.aux = slot;
        return true;
    }
    __device__ void epilogue(const Fp4Item& w, uint32_t taddr, int row) const {
        const int slot = w.aux;
        const int e = c.slot_expert[slot];
        const bool valid = w.m * kGM + row < c.slot_cnt[slot];
        const int rp = (c.poff[slot] / kGM + w.m) * kGM + row;   // padded row
        const float s_a = valid ? c.sa[rp] : 0.f;
        const float tg = c.tscale[e * 3 + 0] * s_a, tu = c.tscale[e * 3 + 1] * s_a;
        __nv_bfloat16* dst = c.h + (size_t)rp * c.f + w.n * 64;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            uint32_t g[16], u[16];
            tmem_ld16(taddr + 16 * j, g);
            tmem_ld16(taddr + 64 + 16 * j, u);
            tmem_ld_wait();
            if (valid) {
                uint32_t packed[8];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float g0 = __uint_as_float(g[i]) * tg, g1 = __uint_as_float(g[i + 1]) * tg;
                    const float u0 = __uint_as_float(u[i]) * tu, u1 = __uint_as_float(u[i + 1]) * tu;
                    const float h0 = g0 / (1.0f + expf(-g0)) * u0;
                    const float h1 = g1 / (1.0f + expf(-g1)) * u1;
                    __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
                    packed[i / 2] = *reinterpret_cast<uint32_t*>(&hb);
                }
                *reinterpret_cast<uint4*>(dst + 16 * j) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                *reinterpret_cast<uint4*>(dst + 16 * j + 8) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
        }
    }
};

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float cc, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(cc), "f"(d)
                 : "memory");
}

// down GEMM: item = (M-tile, N-tile of 128 output columns). mode 0: the shared
// expert's M-tiles (stores); mode 1: the routed experts' M-tiles (adds).
struct Gemm2 {
    PrefillCtx c;
    int NT, KT, mode;
    __device__ int shared_mtiles() const { return (c.T + kGM - 1) / kGM; }
    __device__ int n_items() const {
        const int total = c.meta[2], sh = shared_mtiles();
        return (mode == 0 ? sh : total - sh) * NT;
    }
    __device__ bool item(int i, Fp4Item& w) const {
        const int base = mode == 0 ? c.meta[2] - shared_mtiles() : 0;
        const int mt = base + i / NT, nt = i % NT;
        const int slot = c.mt_slot[mt], m = c.mt_m[mt];
        const int e = c.slot_expert[slot];
        const int rt = c.poff[slot] / kGM + m;
        w.a = c.a2 + (size_t)rt * KT * kGTile;
        w.asf = c.a2sf + (size_t)rt * KT * kGSf;
        w.b = c.w2 + ((size_t)e * NT + nt) * KT * kGTile;
        w.bsf = c.w2sf + ((size_t)e * NT + nt) * KT * kGSf;
        w.kt = KT;
        w.m = m;
        w.n = nt;
        w.aux = slot;
        return true;
    }
    __device__ void epilogue(const Fp4Item& w, uint32_t taddr, int row) const {
        const int slot = w.aux;
        const int e = c.slot_expert[slot];
        const int q = w.m * kGM + row;
        const bool valid = q < c.slot_cnt[slot];
        const int rp = (c.poff[slot] / kGM + w.m) * kGM + row;
        int t = 0;
        float scale = 0.f;
        if (valid) {
            const int p = c.slot_off[slot] + q;
            t = ctx_token(c, p);
            const float wr = p < c.T * c.k ? c.wts[__ldg(c.perm + p)] : 1.0f;
            scale = c.sh[rp] * c.tscale[e * 3 + 2] * wr;
        }
        float* dst = c.out32 + (size_t)t * c.d + w.n * kGN;
#pragma unroll 1
        for (int j = 0; j < kGN / 16; ++j) {
            uint32_t y[16];
            tmem_ld16(taddr + 16 * j, y);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float a0 = __uint_as_float(y[i]) * scale, a1 = __uint_as_float(y[i + 1]) * scale;
                    const float a2 = __uint_as_float(y[i + 2]) * scale, a3 = __uint_as_float(y[i + 3]) * scale;
                    if (mode == 0)
                        *reinterpret_cast<float4*>(dst + 16 * j + i) = make_float4(a0, a1, a2, a3);
                    else
                        red_add_v4(dst + 16 * j + i, a0, a1, a2, a3);
                }
            }
        }
    }
};

__global__ void cast_out_kernel(const float* __restrict__ s, __nv_bfloat16* __restrict__ out,
                                const __nv_bfloat16* __restrict__ residual, size_t n) {
    for (size_t i = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) * 4; i < n; i += (size_t)gridDim.x * blockDim.x * 4) {
        const float4 v = *reinterpret_cast<const float4*>(s + i);
        float o[4] = {v.x, v.y, v.z, v.w};
        __nv_bfloat16 b[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            b[u] = __float2bfloat16_rn(o[u]);
            if (residual != nullptr) b[u] = __float2bfloat16_rn(__bfloat162float(residual[i + u]) + __bfloat162float(b[u]));
        }
        *reinterpret_cast<uint2*>(out + i) = make_uint2(
            (uint32_t)__bfloat16_as_ushort(b[0]) | ((uint32_t)__bfloat16_as_ushort(b[1]) << 16),
            (uint32_t)__bfloat16_as_ushort(b[2]) | ((uint32_t)__bfloat16_as_ushort(b[3]) << 16));
    }
}

// Gate/up weights -> swizzled tiles with gate and up interleaved per 64 rows:
// N-tile nt rows 0..63 = gate rows 64nt.., rows 64..127 = up rows 64nt..
// Down weights -> plain row tiles. One thread per 16 bytes of codes.
__global__ void pack_expert_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                   uint8_t* __restrict__ w1, uint8_t* __restrict__ w1sf, uint8_t* __restrict__ w2,
                                   uint8_t* __restrict__ w2sf, int n_slots, int d, int f, size_t cpm, size_t spm) {
    const int NT1 = 2 * f / kGN, KT1 = d / kGK, NT2 = d / kGN, KT2 = f / kGK;
    const long per_mat16 = (long)cpm / 16;
    const long total = (long)n_slots * 3 * per_mat16;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
        const int e = (int)(i / (3 * per_mat16));
        const int mat = (int)((i / per_mat16) % 3);
        const long byte = (i % per_mat16) * 16;
        const int K = mat < 2 ? d : f;
        const int row = (int)(byte / (K / 2)), col = (int)(byte % (K / 2));
        const int kt = col / 128, j = col % 128;
        const uint8_t* src = codes + ((size_t)e * 3 + mat) * cpm + byte;
        const uint8_t* ssrc = scales + ((size_t)e * 3 + mat) * spm + (size_t)row * (K / 16) + col / 8;
        uint8_t* tile;
        uint8_t* sft;
        int r;
        if (mat < 2) {
            const int nt = row / 64;
            r = (row % 64) + 64 * mat;
            const size_t t = ((size_t)e * NT1 + nt) * KT1 + kt;
            tile = w1 + t * kGTile;
            sft = w1sf + t * kGSf;
        } else {
            const int nt = row / kGN;
            r = row % kGN;
            const size_t t = ((size_t)e * NT2 + nt) * KT2 + kt;
            tile = w2 + t * kGTile;
            sft = w2sf + t * kGSf;
        }
        *reinterpret_cast<uint4*>(tile + swz_offset(r, j)) = *reinterpret_cast<const uint4*>(src);
        sft[r * 16 + j / 8] = ssrc[0];
        sft[r * 16 + j / 8 + 1] = ssrc[1];
    }
}

// Canonical-layout activation quantisation (for the per-step entry point).
template <int EPL>
__global__ void __launch_bounds__(256) act_quant_kernel(const __nv_bfloat16* __restrict__ x, int T, int K,
                                                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                        float* __restrict__ rowscale) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = blockIdx.x * 8 + warp; t < T; t += gridDim.x * 8) {
        for (int k0 = 0; k0 < K; k0 += 32 * EPL) {   // K = 32*EPL*chunks; each chunk is one warp row
            const __nv_bfloat16* xr = x + (size_t)t * K + k0 + lane * EPL;
            float v[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) v[i] = __bfloat162float(xr[i]);
            uint32_t c[EPL / 8];
            uint32_t sb = 0;
            const float s_t = quant_row<EPL>(v, c, sb);
            uint32_t* cd = reinterpret_cast<uint32_t*>(codes + (size_t)t * (K / 2) + (k0 + lane * EPL) / 2);
#pragma unroll
            for (int i = 0; i < EPL / 8; ++i) cd[i] = c[i];
#pragma unroll
            for (int b = 0; b < EPL / 16; ++b) scales[(size_t)t * (K / 16) + (k0 + lane * EPL) / 16 + b] = (sb >> (8 * b)) & 0xffu;
            if (lane == 0 && k0 == 0) rowscale[t] = s_t;
        }
    }
}

}  // namespace

// The row quantisers use 64 (x) and 16 (h) elements per lane: d = 2048, f = 512.
bool prefill_fp4_supported(const Shape& s) {
    return s.wfmt == 0 && s.n_shared == 1 && s.d == 2048 && s.f == 512 && s.E <= 256;
}

size_t prefill_weight_bytes(const Shape& s) {
    const size_t per_expert = (size_t)(2 * s.f / kGN) * (s.d / kGK) * (kGTile + kGSf) +
                              (size_t)(s.d / kGN) * (s.f / kGK) * (kGTile + kGSf);
    return per_expert * s.n_slots();
}

cudaError_t pack_prefill_weights(const Shape& s, const uint8_t* codes, const uint8_t* scales, uint8_t* dst,
                                 cudaStream_t st) {
    const size_t w1 = (size_t)s.n_slots() * (2 * s.f / kGN) * (s.d / kGK) * kGTile;
    const size_t w1sf = (size_t)s.n_slots() * (2 * s.f / kGN) * (s.d / kGK) * kGSf;
    const size_t w2 = (size_t)s.n_slots() * (s.d / kGN) * (s.f / kGK) * kGTile;
    pack_expert_kernel<<<148 * 16, 256, 0, st>>>(codes, scales, dst, dst + w1, dst + w1 + w1sf, dst + w1 + w1sf + w2,
                                                s.n_slots(), s.d, s.f, s.codes_per_matrix(), s.scales_per_matrix());
    return cudaGetLastError();
}

size_t prefill_workspace_bytes(const Shape& s, int Tm) {
    const size_t rows = (size_t)Tm * (s.k + 1) + (size_t)kGM * (s.n_slots() + 1);
    const size_t rt = (rows + kGM - 1) / kGM;
    const size_t a1 = rt * (s.d / kGK) * (kGTile + kGSf);
    const size_t a2 = rt * (s.f / kGK) * (kGTile + kGSf);
    return 256 * 16 + rt * kGM * 4 * 2 + rt * 8 + (s.n_slots() + 2) * 4 + a1 + a2 + rt * kGM * s.f * 2 +
           (size_t)Tm * s.d * 4;
}

cudaError_t prepare_prefill_fp4() {
    cudaError_t e = cudaFuncSetAttribute(fp4_gemm_kernel<Gemm1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fp4_gemm_kernel<Gemm2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

cudaError_t launch_prefill_experts(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                                   const Workspace& ws, uint8_t* pw, int Tm, __nv_bfloat16* out,
                                   const __nv_bfloat16* residual, cudaStream_t st, int* n_launch) {
    // carve the prefill workspace
    const size_t rows = (size_t)Tm * (s.k + 1) + (size_t)kGM * (s.n_slots() + 1);
    const size_t rt = (rows + kGM - 1) / kGM;
    uint8_t* p = pw;
    auto take = [&](size_t n) { uint8_t* r = p; p += (n + 255) / 256 * 256; return r; };
    PrefillCtx c;
    c.perm = ws.perm;
    c.wts = ws.w;
    c.slot_expert = ws.slot_expert;
    c.slot_off = ws.slot_off;
    c.slot_cnt = ws.slot_cnt;
    c.meta = ws.meta;
    c.poff = reinterpret_cast<int*>(take((s.n_slots() + 2) * 4));
    c.mt_slot = reinterpret_cast<int*>(take(rt * 4));
    c.mt_m = reinterpret_cast<int*>(take(rt * 4));
    c.sa = reinterpret_cast<float*>(take(rt * kGM * 4));
    c.sh = reinterpret_cast<float*>(take(rt * kGM * 4));
    c.a1 = take(rt * (s.d / kGK) * kGTile);
    c.a1sf = take(rt * (s.d / kGK) * kGSf);
    c.a2 = take(rt * (s.f / kGK) * kGTile);
    c.a2sf = take(rt * (s.f / kGK) * kGSf);
    c.h = reinterpret_cast<__nv_bfloat16*>(take(rt * kGM * s.f * 2));
    c.out32 = reinterpret_cast<float*>(take((size_t)Tm * s.d * 4));
    c.x = x;
    const size_t w1 = (size_t)s.n_slots() * (2 * s.f / kGN) * (s.d / kGK) * kGTile;
    const size_t w1sf = (size_t)s.n_slots() * (2 * s.f / kGN) * (s.d / kGK) * kGSf;
    const size_t w2 = (size_t)s.n_slots() * (s.d / kGN) * (s.f / kGK) * kGTile;
    c.w1 = L.prefill;
    c.w1sf = L.prefill + w1;
    c.w2 = L.prefill + w1 + w1sf;
    c.w2sf = L.prefill + w1 + w1sf + w2;
    c.tscale = L.tscale;
    c.T = T;
    c.d = s.d;
    c.f = s.f;
    c.E = s.E;
    c.k = s.k;
    plan_kernel<<<1, 256, 0, st>>>(c, ws.meta);
    quant_x_kernel<64><<<148 * 8, 256, 0, st>>>(c);
    Gemm1 g1{c, 2 * s.f / kGN, s.d / kGK};
    fp4_gemm_kernel<Gemm1><<<148, kGThreads, kGSmem, st>>>(g1, ws.status);
    quant_h_kernel<16><<<148 * 8, 256, 0, st>>>(c);
    Gemm2 g2s{c, s.d / kGN, s.f / kGK, 0};
    fp4_gemm_kernel<Gemm2><<<148, kGThreads, kGSmem, st>>>(g2s, ws.status);
    Gemm2 g2r{c, s.d / kGN, s.f / kGK, 1};
    fp4_gemm_kernel<Gemm2><<<148, kGThreads, kGSmem, st>>>(g2r, ws.status);
    const size_t n = (size_t)T * s.d;
    cast_out_kernel<<<148 * 8, 256, 0, st>>>(c.out32, out, residual, n);
    *n_launch += 8;
    return cudaGetLastError();
}

cudaError_t launch_act_quant(const __nv_bfloat16* x, int T, int K, uint8_t* codes, uint8_t* scales, float* rowscale,
                             cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int blocks = (T + 7) / 8 < 148 * 8 ? (T + 7) / 8 : 148 * 8;
    if (K == 2048)
        act_quant_kernel<64><<<blocks, 256, 0, st>>>(x, T, K, codes, scales, rowscale);
    else if (K == 512)
        act_quant_kernel<16><<<blocks, 256, 0, st>>>(x, T, K, codes, scales, rowscale);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace flint

extern "C" flint_status flint_moe_debug_act_quant(const void* x_dev, int T, int K, uint8_t* codes_dev,
                                                  uint8_t* scales_dev, float* rowscale_dev, void* stream) {
    if (T < 0 || (K != 2048 && K != 512)) return FLINT_EINVAL;
    if (T == 0) return FLINT_OK;
    if (x_dev == nullptr || codes_dev == nullptr || scales_dev == nullptr || rowscale_dev == nullptr)
        return FLINT_EINVAL;
    if (((uintptr_t)x_dev & 15u) || ((uintptr_t)codes_dev & 15u) || ((uintptr_t)scales_dev & 3u))
        return FLINT_EINVAL;
    const cudaError_t e = flint::launch_act_quant(static_cast<const __nv_bfloat16*>(x_dev), T, K, codes_dev,
                                                  scales_dev, rowscale_dev, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FLINT_OK : FLINT_ECUDA;
}
