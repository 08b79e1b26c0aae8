// Large-T (prefill) expert projections on the block-scaled FP4 tensor cores.
//
// NVFP4 weights force the FP4 x FP4 tensor-core kind, so the activations that
// enter each projection are quantised to NVFP4 as well (per row: an fp32 scale
// s = amax/2688; per 16 elements: an E4M3 scale E4M3_rne((amax_b/6)/s); codes
// E2M1_rne(v * (1/(E4M3(sb)*s)))). h is kept in fp32 between the two
// projections and quantised from that value. Pipeline for one layer (after
// routing and bucketing):
//   (routing: logits, top-k and each assignment's rank within its expert)
//   plan      offsets, active slots, every slot's rows padded to a multiple
//             of 128 (M-tile table)
//   quant_x   quantise each token's x once and write it into the swizzled A
//             tiles of its k routed experts and of the shared expert
//   gemm1     gate/up: [rows x d] . [2f x d]^T, each 128-column tile holds 64
//             gate and 64 up columns of the same f range, two such tiles per
//             item sharing the A k-tiles; epilogue h = silu(g)*u (fp32,
//             stored blocked so that a warp's stores are contiguous: h_at)
//   quant_h   quantise each fp32 h row into swizzled A tiles of the down GEMM
//             (8 rows per CTA staged in shared memory from coalesced reads)
//   gemm2     down: [rows x f] . [d x f]^T, each M-tile's A tile held in
//             shared memory across its 16 N-tiles; epilogue scales by the routing
//             weight (1 for the shared expert) and stores the contribution in
//             bf16, one row per (token, expert) assignment
//   combine   out[t] = bf16(shared + slot 0 + ... + slot k-1), summed in fp32
//             in that order (deterministic), plus the optional residual
#include <algorithm>

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

// Quantise the warp's row, held as packed bf16 (lane l: EPL consecutive
// elements, EPL/8 uint4). Outputs per lane: EPL/2 code bytes (codes[],
// little-endian words) and EPL/16 scale bytes (packed into sbytes); returns
// the row scale. Values are converted to fp32 on the fly (exactly), so the
// packed row costs EPL/2 registers instead of EPL.
__device__ __forceinline__ void unpack8(const uint4& r, float* v) {
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        v[2 * u] = __low2float(p2[u]);
        v[2 * u + 1] = __high2float(p2[u]);
    }
}

// One 16-element block given its values, the row scale s_t: the block's
// scale byte; its codes into codes[0..1].
__device__ __forceinline__ uint32_t quant_block16(const float (&v)[16], float s_t, uint32_t* codes) {
    float ab = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(v[i]));
    const float ratio = s_t > 0.f ? (ab / 6.0f) / s_t : 0.0f;
    const uint32_t sb = f32_to_e4m3(ratio);
    const float S = e4m3_to_f32(sb) * s_t;
    if (S > 0.f) {
        const float inv = 1.0f / S;
        float q[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = v[i] * inv;
        codes[0] = f32x8_to_e2m1(q);
        codes[1] = f32x8_to_e2m1(q + 8);
    } else {
        codes[0] = 0u;
        codes[1] = 0u;
    }
    return sb;
}

// The same for a row held as fp32 (lane l: EPL consecutive elements).
template <int EPL>
__device__ __forceinline__ float quant_row_f32(const float4 (&raw)[EPL / 4], uint32_t (&codes)[EPL / 8],
                                               uint32_t& sbytes) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(raw[i].x), fabsf(raw[i].y)), fmaxf(fabsf(raw[i].z), fabsf(raw[i].w))));
    const float s_t = warp_max(amax) / 2688.0f;
    sbytes = 0u;
#pragma unroll
    for (int b = 0; b < EPL / 16; ++b) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[4 * i] = raw[4 * b + i].x;
            v[4 * i + 1] = raw[4 * b + i].y;
            v[4 * i + 2] = raw[4 * b + i].z;
            v[4 * i + 3] = raw[4 * b + i].w;
        }
        sbytes |= quant_block16(v, s_t, codes + 2 * b) << (8 * b);
    }
    return s_t;
}

template <int EPL>
__device__ __forceinline__ float quant_row(const uint4 (&raw)[EPL / 8], uint32_t (&codes)[EPL / 8], uint32_t& sbytes) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPL / 8; ++i) {
        float v[8];
        unpack8(raw[i], v);
#pragma unroll
        for (int u = 0; u < 8; ++u) amax = fmaxf(amax, fabsf(v[u]));
    }
    const float amax_t = warp_max(amax);
    const float s_t = amax_t / 2688.0f;
    sbytes = 0u;
#pragma unroll
    for (int b = 0; b < EPL / 16; ++b) {
        float v[16];
        unpack8(raw[2 * b], v);
        unpack8(raw[2 * b + 1], v + 8);
        sbytes |= quant_block16(v, s_t, codes + 2 * b) << (8 * b);
    }
    return s_t;
}

// Write the lane's part of row r of a row tile of blocks (K elements; lane
// owns elements [lane*EPL, (lane+1)*EPL)): codes into the swizzled tile, scales
// after it, of the lane's k-tile block.
template <int EPL>
__device__ __forceinline__ void store_row_swizzled(uint8_t* blocks, int r, int lane,
                                                   const uint32_t (&codes)[EPL / 8], uint32_t sbytes) {
    const int e0 = lane * EPL;                 // first element
    const int kt = e0 / kGK;
    const int j = (e0 % kGK) / 2;              // byte within the 128-byte row of the k-tile
    uint8_t* t = blocks + (size_t)kt * kGBlk;
    if constexpr (EPL >= 32) {
#pragma unroll
        for (int c = 0; c < EPL / 32; ++c)
            *reinterpret_cast<uint4*>(t + swz_offset(r, j + 16 * c)) =
                make_uint4(codes[4 * c], codes[4 * c + 1], codes[4 * c + 2], codes[4 * c + 3]);
    } else {
        *reinterpret_cast<uint2*>(t + swz_offset(r, j)) = make_uint2(codes[0], codes[1]);
    }
    uint8_t* s = t + kGTile + r * 16 + (e0 % kGK) / 16;
    if constexpr (EPL == 64) {
        *reinterpret_cast<uint32_t*>(s) = sbytes;
    } else {
        *s = (uint8_t)sbytes;
    }
}

struct PrefillCtx {
    // routing / bucketing results
    int* perm;                // sorted position -> assignment (written by quant_x)
    const float* wts;
    const int* slot_expert;
    const int* slot_off;
    const int* slot_cnt;
    const int* meta;          // [0] active slots, [2] M-tiles (written by the plan kernel)
    const int* idx;           // [T][k] selected experts
    int* inv;                 // [T*k] rank of assignment t*k+j within its expert, then (quant_x) its bucketed position
    // plan
    int* poff;                // [slots] first padded row of each slot
    int* slot_of;             // [E+1] slot of each active expert
    int* mt_slot;             // [M-tiles] slot of the tile
    int* mt_m;                // [M-tiles] index of the tile within its slot
    int* mt_e;                // [M-tiles] expert of the tile (n_experts: shared)
    // M-tile mt is also row tile mt of the activation buffers (tiles are
    // numbered in padded-row order)
    // activations
    const __nv_bfloat16* x;
    uint8_t* a1;              // gate/up A blocks [row tiles][d/256]
    float* sa;
    float* h;                 // fp32, blocked: see h_at
    uint8_t* a2;              // down A blocks [row tiles][f/256]
    int* prow;                // [padded rows] bucketed position of the row's assignment, -1: padding
    float* yscale;            // [padded rows] s_h * down tensor scale * routing weight
    __nv_bfloat16* y;         // [T*(k+1)][d] weighted contributions by bucketed position
    // weights (blocks)
    const uint8_t* w1;
    const uint8_t* w2;
    const float* tscale;
    int T, d, f, E, k;
};

// Counts -> offsets -> slots -> M-tile table, in one CTA of 256 threads
// (expert e = thread e): the exclusive scan of the per-expert counts gives
// the offsets and the active slots (experts with assignments, in expert
// order, then the shared expert); each slot's rows are padded to whole
// 128-row M-tiles. The counters are zeroed for the next forward.
__global__ void __launch_bounds__(256) scan_plan_kernel(PrefillCtx c, int* __restrict__ ecount,
                                                        int* __restrict__ offsets, int* __restrict__ slot_expert,
                                                        int* __restrict__ slot_off, int* __restrict__ slot_cnt,
                                                        int* __restrict__ meta) {
    griddep_wait();
    __shared__ int wsum[8];
    __shared__ int s_cnt[258], s_exp[258], s_base[258];
    __shared__ int s_ns, s_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = threadIdx.x;
    const int cnt = e < c.E ? ecount[e * kEcountStride] : 0;
    if (e < c.E) ecount[e * kEcountStride] = 0;
    // exclusive scan of (count | active << 20)
    int x = cnt | ((cnt > 0 ? 1 : 0) << 20);
    const int v = x;
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
    const int excl = wsum[warp] + x - v;
    const int off = excl & 0xfffff, slot = excl >> 20;
    if (e < c.E) {
        offsets[e] = off;
        if (cnt > 0) {
            slot_expert[slot] = e;
            slot_off[slot] = off;
            slot_cnt[slot] = cnt;
            s_cnt[slot] = cnt;
            s_exp[slot] = e;
        }
    }
    if (threadIdx.x == 0) {
        const int n_assign = s_total & 0xfffff;
        const int ns = s_total >> 20;
        offsets[c.E] = n_assign;
        slot_expert[ns] = c.E;            // the shared expert: every token, after the routed positions
        slot_off[ns] = c.T * c.k;
        slot_cnt[ns] = c.T;
        s_cnt[ns] = c.T;
        s_exp[ns] = c.E;
        s_ns = ns + 1;
        meta[0] = ns + 1;
        meta[1] = c.T;
    }
    __syncthreads();
    // M-tiles per slot and their exclusive scan (slots 0..255 by thread; a
    // 257th slot, possible only with all 256 experts active, by thread 0)
    const int n_slots = s_ns;
    const int i = threadIdx.x;
    const int mt = i < n_slots ? (s_cnt[i] + kGM - 1) / kGM : 0;
    x = mt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
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
            run += (s_cnt[sl] + kGM - 1) / kGM;
        }
        s_total = run;
    }
    __syncthreads();
    for (int sl = threadIdx.x; sl < n_slots; sl += blockDim.x) {
        const int base = s_base[sl];
        const int m_tiles = (s_cnt[sl] + kGM - 1) / kGM;
        c.poff[sl] = base * kGM;
        c.slot_of[s_exp[sl]] = sl;
        for (int m = 0; m < m_tiles; ++m) {
            c.mt_slot[base + m] = sl;
            c.mt_m[base + m] = m;
            c.mt_e[base + m] = s_exp[sl];
        }
    }
    if (threadIdx.x == 0) meta[2] = s_total;
}

// cp.async (16 bytes, L2 only) into shared memory and its group waits
__device__ __forceinline__ void qx_cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void qx_cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void qx_cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// quant_row on a row staged in shared memory: lane l's chunk i (8 bf16) at
// row[i ^ sw]. The same arithmetic as quant_row and quant_block16: the row
// maximum over all elements, then per 16-element block its maximum, its E4M3
// scale and the codes of v * (1 / (E4M3(sb) * s)); the chunks are read again
// for each pass instead of being held in registers.
template <int EPL>
__device__ __forceinline__ float quant_row_staged(const uint4* row, int sw, uint32_t (&codes)[EPL / 8],
                                                 uint32_t& sbytes) {
    float amax = 0.f;
#pragma unroll 2
    for (int i = 0; i < EPL / 8; ++i) {
        float v[8];
        unpack8(row[i ^ sw], v);
#pragma unroll
        for (int u = 0; u < 8; ++u) amax = fmaxf(amax, fabsf(v[u]));
    }
    const float s_t = warp_max(amax) / 2688.0f;
    sbytes = 0u;
#pragma unroll
    for (int b = 0; b < EPL / 16; ++b) {
        float ab = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[8];
            unpack8(row[(2 * b + h) ^ sw], v);
#pragma unroll
            for (int u = 0; u < 8; ++u) ab = fmaxf(ab, fabsf(v[u]));
        }
        const float ratio = s_t > 0.f ? (ab / 6.0f) / s_t : 0.0f;
        const uint32_t sb = f32_to_e4m3(ratio);
        const float S = e4m3_to_f32(sb) * s_t;
        sbytes |= sb << (8 * b);
        if (S > 0.f) {
            const float inv = 1.0f / S;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[8];
                unpack8(row[(2 * b + h) ^ sw], v);
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] *= inv;
                codes[2 * b + h] = f32x8_to_e2m1(v);
            }
        } else {
            codes[2 * b] = 0u;
            codes[2 * b + 1] = 0u;
        }
    }
    return s_t;
}

// Quantise x[t] once per token (one warp per token) and write the row into
// the A tiles of its k routed experts and of the shared expert (the last
// slot). Padding rows of the tiles are never written: their products are
// discarded by the epilogues. The row is staged in the warp's shared-memory
// slot by cp.async (coalesced: copy i moves the row's 16-byte chunk
// 32 i + lane), which keeps the loads in flight without registers, so that
// kQxCtasPerSm CTAs fit per SM: the kernel is bound by the latency of its
// loads and lookups, and more warps keep more of them in flight. Lane l's
// chunk j sits at slot chunk 8 l + (j ^ (l % 8)), so that the chunk reads of
// 8 consecutive lanes fall in distinct banks. With 3 CTAs per SM and the row
// in registers (80 registers) the warm layer measured 301.1 us; staged, with
// 5 CTAs per SM (48 registers), 296.1 us (6 CTAs: 296.7 us).
constexpr int kQxCtasPerSm = 5;
template <int EPL>
__global__ void __launch_bounds__(256, kQxCtasPerSm) quant_x_kernel(PrefillCtx c) {
    griddep_wait();
    constexpr int NC = EPL / 8;   // 16-byte chunks per lane
    static_assert(NC == 8, "the chunk swizzle assumes 8 chunks per lane");
    __shared__ __align__(16) uint4 xs[8][32 * NC];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = c.d / kGK;
    const int shared_slot = c.meta[0] - 1;
    uint4* slot_rows = xs[warp];
    for (int t = blockIdx.x * 8 + warp; t < c.T; t += gridDim.x * 8) {
        const uint4* src = reinterpret_cast<const uint4*>(c.x + (size_t)t * c.d);
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const int g = i * 32 + lane, L = g / NC, j = g % NC;
            qx_cp_async16(slot_rows + L * NC + (j ^ (L & 7)), src + g);
        }
        qx_cp_async_commit();
        // destination rows, lane j <= k, looked up while the row is in flight
        int my_rp = 0;
        if (lane < c.k) {
            // the assignment's rank within its expert (token_rank_kernel) gives
            // its padded row and its bucketed position
            const int a = t * c.k + lane;
            const int slot = c.slot_of[c.idx[a]];
            const int rank = c.inv[a];
            my_rp = c.poff[slot] + rank;
            const int pos = c.slot_off[slot] + rank;
            c.inv[a] = pos;
            c.perm[pos] = a;
        } else if (lane == c.k) {
            my_rp = c.poff[shared_slot] + t;
        }
        qx_cp_async_wait_all();
        __syncwarp();
        uint32_t codes[EPL / 8];
        uint32_t sb = 0;
        const float s_t = quant_row_staged<EPL>(slot_rows + lane * NC, lane & 7, codes, sb);
        __syncwarp();   // every lane has read the slot before the next token's copies
        for (int j = 0; j <= c.k; ++j) {
            const int rp = __shfl_sync(0xffffffffu, my_rp, j);
            const int rt = rp / kGM, r = rp % kGM;
            store_row_swizzled<EPL>(c.a1 + (size_t)rt * KT * kGBlk, r, lane, codes, sb);
            if (lane == 0) c.sa[rp] = s_t;
        }
    }
}

// h between the two GEMMs, fp32, blocked so that a warp of the gate/up
// epilogue (one accumulator row per lane) stores 512 contiguous bytes: per
// M-tile, per 16-column chunk, per float4 of the chunk, the M-tile's 128 rows
// one after another.
__device__ __forceinline__ float4* h_at(float* h, int f, int mt, int chunk, int q4, int row) {
    return reinterpret_cast<float4*>(h) + ((((size_t)mt * (f / 16) + chunk) * 4 + q4) * kGM + row);
}

constexpr int kQhRows = 2;                       // rows per warp
constexpr int kQhWarps = 4;
constexpr int kQhThreads = 32 * kQhWarps;
constexpr int kQhCtaRows = kQhWarps * kQhRows;   // consecutive rows of one M-tile per CTA
// staged row: 32 chunks of 16 floats, each followed by 4 floats of padding,
// plus 4, so that the chunk reads (one row, lane l at chunk l) fall in
// distinct banks
constexpr int kQhChunkPitch = 20;
constexpr int kQhPitch = 32 * kQhChunkPitch + 4;
constexpr int kQhSmem = kQhCtaRows * kQhPitch * 4;

// Quantise each h row (fp32) into the down GEMM's A tiles and write the down
// GEMM's per-row epilogue data. A CTA takes kQhCtaRows (8) consecutive rows
// of one M-tile, the last CTA the first rows (the gate/up GEMM wrote the high
// rows last, so they are the likeliest still in L2). It reads them from the
// blocked h with every warp load covering four whole 128-byte lines (8 rows
// of one 16-byte piece each), all loads issued before the rows' slot lookups,
// stages them row-major in shared memory, then each warp quantises kQhRows
// rows (lane l: elements 16 l .. 16 l + 15). Small CTAs (64 registers, 21 KB
// of shared memory) let many of them per SM overlap their loads with other
// CTAs' quantisation: 32-row CTAs took 56.9 us (cold), 16-row 42.9 us; 8-row
// CTAs took the warm layer 305.5 -> 301.6 us. Padding rows get prow = -1.
template <int EPL>
__global__ void __launch_bounds__(kQhThreads) quant_h_kernel(PrefillCtx c) {
    griddep_wait();
    static_assert(EPL == 16, "a lane's elements are one 16-column chunk of the row");
    extern __shared__ __align__(16) float qhs[];   // [kQhCtaRows][kQhPitch]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = c.f / kGK;
    const int rb = (gridDim.x - 1 - blockIdx.x) * kQhCtaRows;
    if (rb >= c.meta[2] * kGM) return;
    const int mt = rb / kGM, rin = rb % kGM;
    // thread t loads row t % kQhCtaRows of the CTA's rows, pieces
    // t / kQhCtaRows + kQhStride k
    constexpr int kPer = kQhCtaRows * (512 / 4) / kQhThreads;
    constexpr int kQhStride = kQhThreads / kQhCtaRows;
    const int r_t = threadIdx.x % kQhCtaRows, cq0 = threadIdx.x / kQhCtaRows;
    float4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int cq = cq0 + kQhStride * k;   // chunk * 4 + float4 of the chunk
        v[k] = *h_at(c.h, c.f, mt, cq >> 2, cq & 3, rin + r_t);
    }
    const int row0 = rb + warp * kQhRows, r0 = row0 % kGM;
    const int slot = c.mt_slot[mt], m = c.mt_m[mt];
    // lane i < kQhRows: position and epilogue scale of row row0 + i (-1: padding)
    int p = -1;
    float yscale_w = 0.f;
    if (lane < kQhRows) {
        const int q = m * kGM + r0 + lane;
        if (q < c.slot_cnt[slot]) {
            p = c.slot_off[slot] + q;
            const float wr = p < c.T * c.k ? c.wts[__ldg(c.perm + p)] : 1.0f;
            yscale_w = c.tscale[c.slot_expert[slot] * 3 + 2] * wr;
        }
    }
    uint8_t* blocks = c.a2 + (size_t)mt * KT * kGBlk;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int cq = cq0 + kQhStride * k;
        *reinterpret_cast<float4*>(qhs + r_t * kQhPitch + (cq >> 2) * kQhChunkPitch + (cq & 3) * 4) = v[k];
    }
    __syncthreads();   // the CTA's rows are staged
    float4 raw[kQhRows][EPL / 4];
#pragma unroll
    for (int i = 0; i < kQhRows; ++i)
#pragma unroll
        for (int j = 0; j < EPL / 4; ++j)
            raw[i][j] = *reinterpret_cast<const float4*>(qhs + (warp * kQhRows + i) * kQhPitch + lane * kQhChunkPitch +
                                                         4 * j);
#pragma unroll
    for (int i = 0; i < kQhRows; ++i) {
        const int pi = __shfl_sync(0xffffffffu, p, i);
        const float ys = __shfl_sync(0xffffffffu, yscale_w, i);
        if (pi < 0) {   // padding row: its codes are never read back
            if (lane == 0) c.prow[row0 + i] = -1;
            continue;
        }
        uint32_t codes[EPL / 8];
        uint32_t sb = 0;
        const float s_t = quant_row_f32<EPL>(raw[i], codes, sb);
        store_row_swizzled<EPL>(blocks, r0 + i, lane, codes, sb);
        if (lane == 0) {
            c.prow[row0 + i] = pi;
            c.yscale[row0 + i] = s_t * ys;
        }
    }
}

// gate/up GEMM: item = (M-tile, pair of N-tiles); N-tile nt holds 64 gate
// and 64 up columns of the same f range, so the pair yields h columns
// [128 pair, 128 pair + 128). Both N-tiles share each A k-tile in shared
// memory (the engine's kNB = 2).
struct Gemm1 {
    PrefillCtx c;
    int NT, KT;   // N-tiles (2f/128) and k-tiles (d/256)
    static constexpr int kStages = 4;
    static constexpr int kNB = 2;
    static constexpr int kKPS = 1;          // one A k-tile and the pair's two B k-tiles per stage
    static constexpr bool kBPair = false;
    __device__ int n_items() const { return c.meta[2] * (NT / 2); }
    __device__ void item(int i, Fp4Item& w) const {
        const int np = NT / 2;
        const int mt = i / np, pair = i % np;
        const int e = c.mt_e[mt];
        w.a = c.a1 + (size_t)mt * KT * kGBlk;
        w.b = c.w1 + ((size_t)e * NT + 2 * pair) * KT * kGBlk;
        w.b2 = w.b + (size_t)KT * kGBlk;
        w.kt = KT;
        w.m = mt;
        w.n = pair;
        w.aux = e;
    }
    // Padding rows are computed too (from whatever their tiles hold) and their
    // h rows written; nothing reads them back. No load here feeds a branch,
    // so the prefetch one item ahead does not stall the warp.
    struct Pre {
        float tg, tu;
    };
    __device__ Pre pre(const Fp4Item& w, int row, int) const {
        const float s_a = c.sa[w.m * kGM + row];
        return {c.tscale[w.aux * 3 + 0] * s_a, c.tscale[w.aux * 3 + 1] * s_a};
    }
    static constexpr int kEpiSmemPerWarp = 0;
    __device__ void epilogue_finish() const {}
    // For each N-tile b of the pair: h columns [64 (2 pair + b) + 32 half, +32)
    // from gate accumulator columns 32 half.. and up columns 64 + 32 half..,
    // in two rounds of 16 columns; each round's four tensor-memory loads are
    // issued before its one wait, and the accumulators are released as soon
    // as the second round has been read.
    template <class Release>
    __device__ void epilogue(const Fp4Item& w, const Pre& pr, uint32_t taddr, int row, int half, uint8_t*,
                             Release release) const {
        const float tg = pr.tg, tu = pr.tu;
        // 16-column chunk of (b, r): 8 pair + 4 b + 2 half + r
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            uint32_t g[2][16], u[2][16];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t t = taddr + b * kGN + half * 32 + 16 * r;
                tmem_ld16(t, g[b]);
                tmem_ld16(t + 64, u[b]);
            }
            tmem_ld_wait();
            if (r == 1) release();
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int chunk = 8 * w.n + 4 * b + 2 * half + r;
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    float hv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float gq = __uint_as_float(g[b][i + q]) * tg, uq = __uint_as_float(u[b][i + q]) * tu;
                        // silu(g) * u with the fast exponential and division
                        // (relative error ~1e-6; it can move a later FP4 code
                        // only where h sits on a rounding boundary)
                        hv[q] = __fdividef(gq, 1.0f + __expf(-gq)) * uq;
                    }
                    // the warp's 32 rows write 512 contiguous bytes; the rows
                    // written last are still in L2 when the h quantiser, which
                    // walks the rows from the end, reads them
                    *h_at(c.h, c.f, w.m, chunk, i >> 2, row) = make_float4(hv[0], hv[1], hv[2], hv[3]);
                }
            }
        }
    }
};

// down GEMM epilogue of one (M-tile, N-tile of 128 output columns)
// accumulator, every slot's M-tiles including the shared expert's; run by
// fp4_gemm_resa_kernel through Gemm2R. Each epilogue thread scales its row by
// s_h * tensor scale * routing weight and rounds it to bf16; the warp stages
// its 32 rows x 64 columns in shared memory and writes them, transposed, to
// the rows of their assignments (routed: bucketed position p < T*k; shared:
// T*k + token) with whole 128-byte segments per store.
constexpr int kEpiPitch = 144;   // 128 bytes of a row + 16: conflict-free 16-byte stores
struct Gemm2 {
    PrefillCtx c;
    int NT, KT;
    static constexpr int kEpiSmemPerWarp = 32 * kEpiPitch;
    struct Pre {
        int p;           // bucketed position (shared expert: T*k + token); -1: padding row
        float scale;
    };
    __device__ void epilogue(const Fp4Item& w, const Pre& pr, uint32_t taddr, int row, int half,
                             uint8_t* epi) const {
        const int p = pr.p;
        const float scale = pr.scale;
        const int lane = row & 31;
        uint8_t* srow = epi + lane * kEpiPitch;
        // all four tensor-memory loads in flight before the one wait
        uint32_t y[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(taddr + half * 64 + 16 * j, y + 16 * j);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(y[16 * j + i]) * scale,
                                                         __uint_as_float(y[16 * j + i + 1]) * scale);
                packed[i / 2] = *reinterpret_cast<uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(srow + 32 * j) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<uint4*>(srow + 32 * j + 16) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
        __syncwarp();
        // transposed write-out: each store instruction covers four whole
        // 128-byte row segments (lanes 8r'..8r'+7 take row 4*it + r')
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int r = 4 * it + (lane >> 3), chunk = lane & 7;
            const int pr = __shfl_sync(0xffffffffu, p, r);
            const uint4 v = *reinterpret_cast<const uint4*>(epi + r * kEpiPitch + chunk * 16);
            if (pr >= 0)
                *reinterpret_cast<uint4*>(c.y + (size_t)pr * c.d + w.n * kGN + half * 64 + chunk * 8) = v;
        }
        __syncwarp();
    }
};

// The down GEMM with each M-tile's A tile resident (fp4_gemm_resa_kernel):
// one item per M-tile, its 16 N-tiles in turn; the epilogue is Gemm2's.
struct Gemm2R {
    Gemm2 g;
    static constexpr int kStages = 3;
    static constexpr int kNT = 16;   // d / 128 output column tiles (d = 2048)
    static constexpr int kEpiSmemPerWarp = Gemm2::kEpiSmemPerWarp;
    using Pre = Gemm2::Pre;
    __device__ int n_mtiles() const { return g.c.meta[2]; }
    __device__ const uint8_t* a_blocks(int mt) const { return g.c.a2 + (size_t)mt * kRKT * kGBlk; }
    __device__ const uint8_t* b_blocks(int mt, int n) const {
        return g.c.w2 + ((size_t)__ldg(g.c.mt_e + mt) * kNT + n) * kRKT * kGBlk;
    }
    __device__ Pre pre(int mt, int row, int) const {
        const int rp = mt * kGM + row;
        return {g.c.prow[rp], g.c.yscale[rp]};
    }
    __device__ void epilogue(int mt, int n, const Pre& pr, uint32_t taddr, int row, int half, uint8_t* epi) const {
        Fp4Item w;
        w.a = w.b = w.b2 = nullptr;
        w.kt = kRKT;
        w.m = mt;
        w.n = n;
        w.aux = 0;
        g.epilogue(w, pr, taddr, row, half, epi);
    }
};

// out[t] = bf16(y[shared] + y[slot 0] + ... + y[slot k-1]) summed in fp32 in
// that order; with a residual, out = bf16(residual + that bf16 value). One
// warp per token, 16 columns per lane per step; every load of a step is
// issued before the first add.
__global__ void __launch_bounds__(256) combine_kernel(PrefillCtx c, __nv_bfloat16* __restrict__ out,
                                                      const __nv_bfloat16* __restrict__ residual) {
    griddep_wait();
    // one CTA per token, 8 columns per thread: every contribution's load is
    // issued before the first is used
    const int t = blockIdx.x, col = threadIdx.x * 8;
    if (t >= c.T || col >= c.d) return;
    uint4 r[9];
    r[0] = __ldcs(reinterpret_cast<const uint4*>(c.y + ((size_t)c.T * c.k + t) * c.d + col));
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j < c.k) r[j + 1] = __ldcs(reinterpret_cast<const uint4*>(c.y + (size_t)__ldg(c.inv + t * c.k + j) * c.d + col));
    // shared + slot 0 + ... + slot k-1, in that order, in fp32
    float acc[8];
    unpack8(r[0], acc);
#pragma unroll
    for (int j = 1; j <= 8; ++j) {
        if (j <= c.k) {
            float v[8];
            unpack8(r[j], v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += v[i];
        }
    }
    uint32_t o[4];
    if (residual != nullptr) {
        float rv[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(residual + (size_t)t * c.d + col)), rv);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const __nv_bfloat16 b0 = __float2bfloat16_rn(rv[2 * u] + __bfloat162float(__float2bfloat16_rn(acc[2 * u])));
            const __nv_bfloat16 b1 =
                __float2bfloat16_rn(rv[2 * u + 1] + __bfloat162float(__float2bfloat16_rn(acc[2 * u + 1])));
            o[u] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const __nv_bfloat16 b0 = __float2bfloat16_rn(acc[2 * u]), b1 = __float2bfloat16_rn(acc[2 * u + 1]);
            o[u] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
        }
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * c.d + col) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Gate/up weights -> blocks (swizzled tile + scales) with gate and up
// interleaved per 64 rows: N-tile nt rows 0..63 = gate rows 64nt.., rows
// 64..127 = up rows 64nt.. Down weights -> plain row tiles of blocks. One
// thread per 16 bytes of codes.
__global__ void pack_expert_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                   uint8_t* __restrict__ w1, uint8_t* __restrict__ w2, int n_slots, int d, int f,
                                   size_t cpm, size_t spm) {
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
        uint8_t* blk;
        int r;
        if (mat < 2) {
            const int nt = row / 64;
            r = (row % 64) + 64 * mat;
            blk = w1 + (((size_t)e * NT1 + nt) * KT1 + kt) * kGBlk;
        } else {
            const int nt = row / kGN;
            r = row % kGN;
            blk = w2 + (((size_t)e * NT2 + nt) * KT2 + kt) * kGBlk;
        }
        *reinterpret_cast<uint4*>(blk + swz_offset(r, j)) = *reinterpret_cast<const uint4*>(src);
        blk[kGTile + r * 16 + j / 8] = ssrc[0];
        blk[kGTile + r * 16 + j / 8 + 1] = ssrc[1];
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
            uint4 raw[EPL / 8];
#pragma unroll
            for (int i = 0; i < EPL / 8; ++i) raw[i] = *reinterpret_cast<const uint4*>(xr + 8 * i);
            uint32_t c[EPL / 8];
            uint32_t sb = 0;
            const float s_t = quant_row<EPL>(raw, c, sb);
            uint32_t* cd = reinterpret_cast<uint32_t*>(codes + (size_t)t * (K / 2) + (k0 + lane * EPL) / 2);
#pragma unroll
            for (int i = 0; i < EPL / 8; ++i) cd[i] = c[i];
#pragma unroll
            for (int b = 0; b < EPL / 16; ++b) scales[(size_t)t * (K / 16) + (k0 + lane * EPL) / 16 + b] = (sb >> (8 * b)) & 0xffu;
            if (lane == 0 && k0 == 0) rowscale[t] = s_t;
        }
    }
}

// NVFP4 quantisation of a bf16 weight matrix with one fp32 tensor scale: the
// amax of the matrix (fp32 bits, atomically maxed: non-negative floats order
// as their bit patterns), then one thread per 16-element block, then the
// tensor scale written over the amax.
__global__ void __launch_bounds__(256) weight_amax_kernel(const __nv_bfloat16* __restrict__ w, long n8,
                                                          uint32_t* __restrict__ amax_bits) {
    float m = 0.f;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n8; i += (long)gridDim.x * blockDim.x) {
        float v[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(w) + i), v);
#pragma unroll
        for (int u = 0; u < 8; ++u) m = fmaxf(m, fabsf(v[u]));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax_bits, __float_as_uint(m));
}

__global__ void __launch_bounds__(256) weight_quant_kernel(const __nv_bfloat16* __restrict__ w, long n_blocks,
                                                           const uint32_t* __restrict__ amax_bits,
                                                           uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    const float s = __uint_as_float(*amax_bits) / 2688.0f;
    for (long b = blockIdx.x * (long)blockDim.x + threadIdx.x; b < n_blocks; b += (long)gridDim.x * blockDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(w + b * 16);
        float v[16];
        unpack8(__ldg(src), v);
        unpack8(__ldg(src + 1), v + 8);
        uint32_t c[2];
        const uint32_t sb = quant_block16(v, s, c);
        *reinterpret_cast<uint2*>(codes + b * 8) = make_uint2(c[0], c[1]);
        scales[b] = (uint8_t)sb;
    }
}

__global__ void weight_scale_kernel(float* tensor_scale) {
    *tensor_scale = __uint_as_float(*reinterpret_cast<const uint32_t*>(tensor_scale)) / 2688.0f;
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
    const size_t w1 = (size_t)s.n_slots() * (2 * s.f / kGN) * (s.d / kGK) * kGBlk;
    pack_expert_kernel<<<148 * 16, 256, 0, st>>>(codes, scales, dst, dst + w1, s.n_slots(), s.d, s.f,
                                                s.codes_per_matrix(), s.scales_per_matrix());
    return cudaGetLastError();
}

size_t prefill_workspace_bytes(const Shape& s, int Tm) {
    const size_t rows = (size_t)Tm * (s.k + 1) + (size_t)kGM * (s.n_slots() + 1);
    const size_t rt = (rows + kGM - 1) / kGM;
    const size_t a1 = rt * (s.d / kGK) * (kGTile + kGSf);
    const size_t a2 = rt * (s.f / kGK) * (kGTile + kGSf);
    return 256 * 16 + rt * kGM * 4 * 3 + rt * 16 + (s.n_slots() + 2) * 4 * 2 + a1 + a2 + rt * kGM * s.f * 4 +
           (size_t)Tm * (s.k + 1) * s.d * 2;
}

cudaError_t prepare_prefill_fp4() {
    cudaError_t e = cudaFuncSetAttribute(fp4_gemm_kernel<Gemm1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fp4_gemm_smem<Gemm1>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fp4_gemm_resa_kernel<Gemm2R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 fp4_gemm_resa_smem<Gemm2R>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(quant_h_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQhSmem);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

cudaError_t launch_prefill_experts(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                                   const Workspace& ws, uint8_t* pw, int Tm, __nv_bfloat16* out,
                                   const __nv_bfloat16* residual, cudaStream_t st, int* n_launch,
                                   const cudaEvent_t* marks) {
    // marks[j] is the forward's profiling mark j+1; marks[1..5] are recorded
    // after quant_x, gemm1, quant_h, gemm2 and the cast (when not null)
    auto mark = [&](int i) {
        if (marks != nullptr) cudaEventRecord(marks[i], st);
    };
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
    c.idx = ws.idx;
    c.inv = ws.inv;
    c.poff = reinterpret_cast<int*>(take((s.n_slots() + 2) * 4));
    c.slot_of = reinterpret_cast<int*>(take((s.n_slots() + 2) * 4));
    c.mt_slot = reinterpret_cast<int*>(take(rt * 4));
    c.mt_m = reinterpret_cast<int*>(take(rt * 4));
    c.mt_e = reinterpret_cast<int*>(take(rt * 4));
    c.sa = reinterpret_cast<float*>(take(rt * kGM * 4));
    c.prow = reinterpret_cast<int*>(take(rt * kGM * 4));
    c.yscale = reinterpret_cast<float*>(take(rt * kGM * 4));
    c.a1 = take(rt * (s.d / kGK) * kGBlk);
    c.a2 = take(rt * (s.f / kGK) * kGBlk);
    c.h = reinterpret_cast<float*>(take(rt * kGM * s.f * 4));
    c.y = reinterpret_cast<__nv_bfloat16*>(take((size_t)Tm * (s.k + 1) * s.d * 2));
    c.x = x;
    const size_t w1 = (size_t)s.n_slots() * (2 * s.f / kGN) * (s.d / kGK) * kGBlk;
    c.w1 = L.prefill;
    c.w2 = L.prefill + w1;
    c.tscale = L.tscale;
    c.T = T;
    c.d = s.d;
    c.f = s.f;
    c.E = s.E;
    c.k = s.k;
    // every kernel of the chain is launched with programmatic serialisation
    // and waits for its predecessor at its first statement (pdl.cuh); the
    // overlapped launches took the layer 319.3 -> 305.3 us
    cudaError_t e = launch_pdl(scan_plan_kernel, dim3(1), dim3(256), 0, st, c, ws.ecount, ws.offsets,
                               ws.slot_expert, ws.slot_off, ws.slot_cnt, ws.meta);
    if (e == cudaSuccess)
        e = launch_pdl(quant_x_kernel<64>, dim3(std::min((T + 7) / 8, 148 * kQxCtasPerSm)), dim3(256), 0, st, c);
    mark(1);
    Gemm1 g1{c, 2 * s.f / kGN, s.d / kGK};
    if (e == cudaSuccess)
        e = launch_pdl(fp4_gemm_kernel<Gemm1>, dim3(148), dim3(kGThreads), fp4_gemm_smem<Gemm1>(), st, g1, ws.status);
    mark(2);
    static_assert(kGM % kQhCtaRows == 0, "a CTA's rows stay inside one M-tile");
    if (e == cudaSuccess)
        e = launch_pdl(quant_h_kernel<16>, dim3((unsigned)(rt * kGM / kQhCtaRows)), dim3(kQhThreads), kQhSmem, st, c);
    mark(3);
    static_assert(Gemm2R::kNT * kGN == 2048 && kRKT * kGK == 512, "the Flint shape (d = 2048, f = 512)");
    Gemm2R g2{Gemm2{c, s.d / kGN, s.f / kGK}};
    if (e == cudaSuccess)
        e = launch_pdl(fp4_gemm_resa_kernel<Gemm2R>, dim3(148), dim3(kGThreads), fp4_gemm_resa_smem<Gemm2R>(), st, g2,
                       ws.status);
    mark(4);
    // one CTA per token, 8 columns per thread
    if (e == cudaSuccess) e = launch_pdl(combine_kernel, dim3(T), dim3(s.d / 8), 0, st, c, out, residual);
    mark(5);
    *n_launch += 6;
    return e;
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

extern "C" flint_status flint_moe_quantize_nvfp4(const void* w_dev, int R, int K, uint8_t* codes_dev,
                                                 uint8_t* scales_dev, float* tensor_scale_dev, void* stream) {
    using namespace flint;
    if (R < 1 || K < 16 || K % 16 != 0) return FLINT_EINVAL;
    if (w_dev == nullptr || codes_dev == nullptr || scales_dev == nullptr || tensor_scale_dev == nullptr)
        return FLINT_EINVAL;
    if (((uintptr_t)w_dev & 15u) || ((uintptr_t)codes_dev & 7u) || ((uintptr_t)tensor_scale_dev & 3u))
        return FLINT_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long n = (long)R * K;
    const auto* w = static_cast<const __nv_bfloat16*>(w_dev);
    uint32_t* amax = reinterpret_cast<uint32_t*>(tensor_scale_dev);
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return FLINT_ECUDA;
    const long n8 = n / 8, nb = n / 16;
    const int g1 = (int)std::min<long>((n8 + 255) / 256, 148L * 8);
    const int g2 = (int)std::min<long>((nb + 255) / 256, 148L * 16);
    weight_amax_kernel<<<g1, 256, 0, st>>>(w, n8, amax);
    weight_quant_kernel<<<g2, 256, 0, st>>>(w, nb, amax, codes_dev, scales_dev);
    weight_scale_kernel<<<1, 1, 0, st>>>(tensor_scale_dev);
    return cudaGetLastError() == cudaSuccess ? FLINT_OK : FLINT_ECUDA;
}
