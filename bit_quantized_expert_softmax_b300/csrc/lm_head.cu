// The 4-bit output head (lm_head) and its sampling front-end.
//
// The Flint blog ("Recursive Flint 40B-A2.5B", section "The quantisation
// recipe is the most transferable part") quantises the output layer to 4 bits
// because, with ~2.5B active parameters per token, it is a large share of the
// bytes read for every token: decoding it is a GEMV that streams ~169 MB of
// NVFP4 weights (146k rows x 2048) for a handful of tokens, so it is bound by
// HBM. Its serving defaults are temperature 1.0, top-p 0.95, top-k 20 (section
// "The three scores, and the footnotes that come with them", Sampling bullet).
//
// head_gemv_kernel: one CTA of 12 warps per SM. Warp w of CTA b owns the
// 8-row units b*12 + w, + 12*G, ... of the head (the tiled layout: one unit is
// d/128 tiles of 8 rows x 128 K, 512 bytes of codes and 64 of scales each) and
// keeps two register chunks of 8 tiles: while one chunk is decoded and
// multiplied, the next chunk's 16-byte loads are in flight. The MMA is
// m16n8k16 with the tokens as its 16 A rows (x as fp16, scaled per token by a
// power of two, staged once per CTA) and 8 weight rows as B, so each warp
// owns whole rows and needs no cross-warp reduction.
//
// head_sample_kernel: grid (parts, T), 256 threads per CTA. Each CTA takes
// the top-k of a 2048-logit slice (8 per thread, in registers; a round's
// winner found by warp reductions and one 64-bit shared atomic max per warp);
// the last CTA of a token merges the parts' candidates into the token's top-k
// and draws (see sample_from_topk).
#include "kernels.cuh"
#include "pdl.cuh"
#include "tiles.cuh"

namespace flint {

namespace {

constexpr int kHeadThreads = 384;   // 12 warps
constexpr int kHeadWarps = kHeadThreads / 32;
constexpr int kHeadChunk = 8;       // tiles per register chunk

struct HeadArgs {
    const uint8_t* codes;   // tiled [V/8][d/128][512]
    const uint8_t* scales;  // tiled [V/8][d/128][64]
    float tscale;
    const __nv_bfloat16* x; // [T][d]
    float* logits;          // [T][V]
    int T, d, V;
};

struct HeadChunk {
    uint4 w[kHeadChunk];
    uint2 s[kHeadChunk];
};

__device__ __forceinline__ void head_load(HeadChunk& ch, const HeadArgs& a, int unit, int kc, int KT, int lane) {
    const int g = lane >> 2;
    const size_t base = (size_t)unit * KT + kc;
#pragma unroll
    for (int i = 0; i < kHeadChunk; ++i) {
        if (kc + i < KT) {
            ch.w[i] = ldg_nc_v4(a.codes + (base + i) * 512 + lane * 16);
            ch.s[i] = ldg_nc_v2(a.scales + (base + i) * 64 + g * 8);
        }
    }
}

// acc += x[tokens] . W[8 rows]^T over the chunk's tiles. Lane (g, c): A
// fragment = token g's fp16 x at its K positions (zero for g >= T), B fragment
// = weight row g decoded from the lane's 16 code bytes and 8 scale bytes.
// Even and odd k-steps go to two accumulators (two independent MMA chains).
__device__ __forceinline__ void head_compute(const HeadChunk& ch, int kc, int KT, const __half* xs, int c,
                                             float (&acc)[4], float (&acc2)[4]) {
#pragma unroll
    for (int i = 0; i < kHeadChunk; ++i) {
        if (kc + i < KT) {
            uint32_t xa[16];
            if (xs != nullptr) {
                const uint4* xp = reinterpret_cast<const uint4*>(xs + (kc + i) * 128 + c * 32);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = xp[q];
                    xa[4 * q + 0] = v.x;
                    xa[4 * q + 1] = v.y;
                    xa[4 * q + 2] = v.z;
                    xa[4 * q + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) xa[q] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {   // code word j: steps 2j, 2j+1
                uint32_t r0, r1, r2, r3;
                e2m1x8_to_f16x2(u4_get(ch.w[i], j), r0, r1, r2, r3);
                const uint32_t sw = u2_get(ch.s[i], j >> 1) >> ((j & 1) * 16);
                const uint32_t s2 = e4m3x2_to_f16x2(sw);
                const uint32_t sa = bcast_lo(s2), sb = bcast_hi(s2);
                mma_16816(acc, xa[4 * j], 0u, xa[4 * j + 1], 0u, hmul2_u(r0, sa), hmul2_u(r1, sa));
                mma_16816(acc2, xa[4 * j + 2], 0u, xa[4 * j + 3], 0u, hmul2_u(r2, sb), hmul2_u(r3, sb));
            }
        }
    }
}

__device__ __forceinline__ void head_store(const HeadArgs& a, int unit, int g, int c, float (&acc)[4],
                                           float (&acc2)[4], const float* xinv) {
    if (g < a.T) {
        const float sc = a.tscale * xinv[g];
        *reinterpret_cast<float2*>(a.logits + (size_t)g * a.V + (size_t)unit * 8 + 2 * c) =
            make_float2((acc[0] + acc2[0]) * sc, (acc[1] + acc2[1]) * sc);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = acc2[j] = 0.f;
}

__global__ void __launch_bounds__(kHeadThreads, 1) head_gemv_kernel(HeadArgs a) {
    griddep_wait();
    extern __shared__ __align__(16) uint8_t hsm[];
    __half* x16 = reinterpret_cast<__half*>(hsm);                              // [T][d]
    float* xinv = reinterpret_cast<float*>(hsm + (size_t)a.T * a.d * 2);      // [kHeadMaxT]
    float* part = xinv + kHeadMaxT;                                            // [kHeadWarps]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KT = a.d >> 7;
    const int n_units = a.V >> 3;
    const int nc = (KT + kHeadChunk - 1) / kHeadChunk;   // chunks per unit
    const int W = gridDim.x * kHeadWarps;
    const int gw = blockIdx.x * kHeadWarps + warp;
    const int total = gw < n_units ? ((n_units - 1 - gw) / W + 1) * nc : 0;   // this warp's chunks
    HeadChunk A, B;
    if (total > 0) head_load(A, a, gw, 0, KT, lane);   // in flight while x is staged
    // x as fp16 with a power-of-two scale per token, fragment-permuted
    for (int t = 0; t < a.T; ++t) {
        const __nv_bfloat16* xr = a.x + (size_t)t * a.d;
        float amax = 0.f;
        for (int i = threadIdx.x * 4; i < a.d; i += kHeadThreads * 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(xr + i);
            const float2 p0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
            const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(p0.x), fabsf(p0.y)), fmaxf(fabsf(p1.x), fabsf(p1.y))));
        }
        amax = warp_max(amax);
        if (lane == 0) part[warp] = amax;
        __syncthreads();
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < kHeadWarps; ++w) m = fmaxf(m, part[w]);
        const float mult = f16_range_mult(m);
        __half2* row = reinterpret_cast<__half2*>(x16 + (size_t)t * a.d);
        for (int i = threadIdx.x * 4; i < a.d; i += kHeadThreads * 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(xr + i);
            const float2 p0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
            const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
            __half2* tile = row + ((i & ~127) >> 1);
            tile[kperm_pos(i & 127) >> 1] = __floats2half2_rn(p0.x * mult, p0.y * mult);
            tile[kperm_pos((i & 127) + 2) >> 1] = __floats2half2_rn(p1.x * mult, p1.y * mult);
        }
        if (threadIdx.x == 0) xinv[t] = 1.0f / mult;
        __syncthreads();
    }
    const __half* xs = g < a.T ? x16 + (size_t)g * a.d : nullptr;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    // chunk q of this warp: unit gw + (q / nc) * W, tiles from (q % nc) * kHeadChunk;
    // the two register chunks alternate so that one is loading while the
    // other is computed
    for (int q = 0; q < total;) {
        if (q + 1 < total) head_load(B, a, gw + ((q + 1) / nc) * W, ((q + 1) % nc) * kHeadChunk, KT, lane);
        head_compute(A, (q % nc) * kHeadChunk, KT, xs, c, acc, acc2);
        if (q % nc == nc - 1) head_store(a, gw + (q / nc) * W, g, c, acc, acc2, xinv);
        if (++q >= total) break;
        if (q + 1 < total) head_load(A, a, gw + ((q + 1) / nc) * W, ((q + 1) % nc) * kHeadChunk, KT, lane);
        head_compute(B, (q % nc) * kHeadChunk, KT, xs, c, acc, acc2);
        if (q % nc == nc - 1) head_store(a, gw + (q / nc) * W, g, c, acc, acc2, xinv);
        ++q;
    }
}

// ---------------------------------------------------------------------------
// sampling front-end
// ---------------------------------------------------------------------------
constexpr int kSampleThreads = 256;
constexpr int kSamplePer = 8;                                  // entries per thread
constexpr int kSampleSlice = kSampleThreads * kSamplePer;      // logits per part

struct SampleArgs {
    const float* logits;   // [T][V]
    int T, V;
    float temperature;
    int k;                 // top-k (1..32)
    float top_p;
    const float* u;        // [T] uniforms in [0, 1)
    int* tokens;           // [T]
    int* topk_idx;         // [T][k] or null
    uint32_t* cand_key;    // [kHeadMaxT][parts][32] order keys of the parts' candidates
    uint32_t* cand_idx;
    unsigned int* counters;   // [kHeadMaxT], zero between calls
    uint32_t* status;
    int parts;
};

// Order-preserving unsigned key of a float (-0 folded onto +0; NaN ranks
// below -inf), and its inverse.
__device__ __forceinline__ uint32_t order_key(float x) {
    if (isnan(x)) return 0u;
    const uint32_t b = __float_as_uint(x + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-K of the CTA's 256 x kSamplePer entries (key 0 with index 0xffffffff:
// empty), by descending key, then ascending index. Each round every warp
// reduces its threads' current bests (max key, then min index among the
// lanes holding it), one 64-bit atomic max per warp picks the CTA's winner,
// and only the thread that held it rescans its entries. sel_key/sel_idx
// (shared, K entries) receive the selections in order.
__device__ __forceinline__ void cta_topk(uint32_t (&key)[kSamplePer], uint32_t (&idx)[kSamplePer], int K,
                                         unsigned long long* best3, uint32_t* sel_key, uint32_t* sel_idx) {
    const int lane = threadIdx.x & 31;
    uint32_t bk = 0u, bi = 0xffffffffu;
    int bs = -1;
    auto rescan = [&]() {
        bk = 0u;
        bi = 0xffffffffu;
        bs = -1;
#pragma unroll
        for (int i = 0; i < kSamplePer; ++i) {
            if (key[i] > bk || (key[i] == bk && idx[i] < bi)) {
                bk = key[i];
                bi = idx[i];
                bs = i;
            }
        }
    };
    rescan();
    if (threadIdx.x < 3) best3[threadIdx.x] = 0ull;
    __syncthreads();
#pragma unroll 1
    for (int j = 0; j < K; ++j) {
        // round j uses best3[j % 3]; the one for round j + 1 was last read in
        // round j - 2, before round j - 1's barrier, so it can be cleared now
        if (threadIdx.x == 0) best3[(j + 1) % 3] = 0ull;
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t wi = __reduce_min_sync(0xffffffffu, bk == wk ? bi : 0xffffffffu);
        if (lane == 0) atomicMax(best3 + j % 3, ((unsigned long long)wk << 32) | (unsigned long long)(~wi));
        __syncthreads();
        const unsigned long long w = best3[j % 3];
        const uint32_t ck = (uint32_t)(w >> 32), ci = ~(uint32_t)w;
        if (threadIdx.x == 0) {
            sel_key[j] = ck;
            sel_idx[j] = ci;
        }
        if (bs >= 0 && bk == ck && bi == ci) {
#pragma unroll
            for (int i = 0; i < kSamplePer; ++i) {
                if (i == bs) {
                    key[i] = 0u;
                    idx[i] = 0xffffffffu;
                }
            }
            rescan();
        }
    }
    __syncthreads();
}

// The draw from a token's top-K (lane j < K of the calling warp holds
// selection j, descending): softmax over them at the temperature, the
// smallest prefix whose probability reaches top_p (a member is kept while the
// sum before it is below top_p), then the first kept member whose cumulative
// probability exceeds u times the kept total.
__device__ __forceinline__ int sample_from_topk(float sv, int si, int K, float temperature, float top_p, float u) {
    const int lane = threadIdx.x & 31;
    if (temperature <= 0.f) return __shfl_sync(0xffffffffu, si, 0);
    const float v0 = __shfl_sync(0xffffffffu, sv, 0);
    const float e = lane < K ? expf((sv - v0) / temperature) : 0.f;
    const float p = e / warp_sum(e);
    float cum = p;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o) cum += y;
    }
    float excl = __shfl_up_sync(0xffffffffu, cum, 1);
    if (lane == 0) excl = 0.f;
    const bool keep = lane < K && (lane == 0 || excl < top_p);
    const int m = __popc(__ballot_sync(0xffffffffu, keep));
    const float Z = __shfl_sync(0xffffffffu, cum, m - 1);
    const unsigned hit = __ballot_sync(0xffffffffu, lane < m && cum > u * Z);
    const int r = hit != 0u ? __ffs(hit) - 1 : m - 1;
    return __shfl_sync(0xffffffffu, si, r);
}

// grid (parts, T): CTA (p, t) takes the top-K of logits [p*2048, (p+1)*2048)
// of token t; the last CTA of the token merges the parts' candidates and draws.
__global__ void __launch_bounds__(kSampleThreads) head_sample_kernel(SampleArgs a) {
    griddep_wait();
    __shared__ unsigned long long best3[3];
    __shared__ uint32_t sel_key[32], sel_idx[32];
    __shared__ int s_last;
    const int part = blockIdx.x, t = blockIdx.y;
    const int K = a.temperature > 0.f ? min(a.k, a.V) : 1;
    const float* L = a.logits + (size_t)t * a.V;
    const int lo = part * kSampleSlice, hi = min(a.V, lo + kSampleSlice);
    uint32_t key[kSamplePer], idx[kSamplePer];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kSamplePer; ++i) {
        const int e = lo + threadIdx.x + kSampleThreads * i;
        if (e < hi) {
            const float x = __ldcg(L + e);
            bad |= isnan(x);
            key[i] = order_key(x);
            idx[i] = (uint32_t)e;
        } else {
            key[i] = 0u;
            idx[i] = 0xffffffffu;
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(a.status, kStatusNonFiniteLogit);
    cta_topk(key, idx, K, best3, sel_key, sel_idx);
    const size_t cbase = ((size_t)t * a.parts + part) * 32;
    if (threadIdx.x < K) {
        a.cand_key[cbase + threadIdx.x] = sel_key[threadIdx.x];
        a.cand_idx[cbase + threadIdx.x] = sel_idx[threadIdx.x];
    }
    // the last part of the token to finish merges all parts' candidates
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.counters + t, 1u) == (unsigned)(a.parts - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int n = a.parts * K;   // <= kSampleSlice (checked by the launcher)
#pragma unroll
    for (int i = 0; i < kSamplePer; ++i) {
        const int e = threadIdx.x + kSampleThreads * i;
        if (e < n) {
            const int pp = e / K, j = e - pp * K;
            const size_t o = ((size_t)t * a.parts + pp) * 32 + j;
            key[i] = __ldcg(a.cand_key + o);
            idx[i] = __ldcg(a.cand_idx + o);
        } else {
            key[i] = 0u;
            idx[i] = 0xffffffffu;
        }
    }
    cta_topk(key, idx, K, best3, sel_key, sel_idx);
    if (threadIdx.x == 0) a.counters[t] = 0u;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const float sv = lane < K ? key_value(sel_key[lane]) : -INFINITY;
        const int si = lane < K ? (int)sel_idx[lane] : -1;
        const int token = sample_from_topk(sv, si, K, a.temperature, a.top_p, a.u[t]);
        if (a.topk_idx != nullptr && lane < K) a.topk_idx[(size_t)t * a.k + lane] = si;
        if (lane == 0) a.tokens[t] = token;
    }
}

}  // namespace

size_t head_smem_bytes(int T, int d) {
    return (size_t)T * d * 2 + (size_t)(kHeadMaxT + kHeadWarps) * sizeof(float);
}

cudaError_t prepare_head() {
    const cudaError_t e = cudaFuncSetAttribute(head_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)head_smem_bytes(kHeadMaxT, kHeadMaxD));
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

cudaError_t launch_head_gemv(const uint8_t* codes, const uint8_t* scales, float tscale, const __nv_bfloat16* x,
                             int T, int d, int V, float* logits, int n_sms, cudaStream_t st) {
    if (T < 1 || T > kHeadMaxT || d % 128 != 0 || d > kHeadMaxD || V % 8 != 0 || V <= 0)
        return cudaErrorInvalidValue;
    HeadArgs a{codes, scales, tscale, x, logits, T, d, V};
    return launch_pdl(head_gemv_kernel, dim3(n_sms), dim3(kHeadThreads), head_smem_bytes(T, d), st, a);
}

int head_sample_parts(int V) { return (V + kSampleSlice - 1) / kSampleSlice; }

bool head_sample_supported(int V, int top_k) {
    return top_k >= 1 && top_k <= 32 && V >= 1 && (size_t)head_sample_parts(V) * top_k <= (size_t)kSampleSlice;
}

cudaError_t launch_head_sample(const float* logits, int T, int V, float temperature, int top_k, float top_p,
                               const float* u, int* tokens, int* topk_idx, const HeadScratch& hs, uint32_t* status,
                               cudaStream_t st) {
    if (T < 1 || T > kHeadMaxT || !head_sample_supported(V, top_k)) return cudaErrorInvalidValue;
    SampleArgs a;
    a.logits = logits;
    a.T = T;
    a.V = V;
    a.temperature = temperature;
    a.k = top_k;
    a.top_p = top_p;
    a.u = u;
    a.tokens = tokens;
    a.topk_idx = topk_idx;
    a.cand_key = hs.cand_key;
    a.cand_idx = hs.cand_idx;
    a.counters = hs.counters;
    a.status = status;
    a.parts = head_sample_parts(V);
    return launch_pdl(head_sample_kernel, dim3(a.parts, T), dim3(kSampleThreads), 0, st, a);
}

}  // namespace flint
