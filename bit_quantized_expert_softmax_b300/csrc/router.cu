// Router (logits, top-k, renormalised softmax), fp16 staging of the hidden
// states, and token -> expert bucketing.
//
// Structure from the Flint blog ("Recursive Flint 40B-A2.5B", section "The
// architecture is an argument about memory bandwidth", Sparsity bullet): 256
// routed experts, 6 chosen per token, one always-on shared expert. The
// routing rule: fp32 logits, the k largest (ties: lower expert index),
// softmax renormalised over the chosen k.
#include <float.h>

#include "kernels.cuh"
#include "topk.cuh"

namespace flint {

namespace {

constexpr int kRouterThreads = 256;   // 8 warps: 2 experts x 4 K-quarters
constexpr int kMaxKIt = 8;            // d <= 4096 for the register-resident router row

// ---------------------------------------------------------------------------
// fp16 staging of one token: per-token power-of-two scale, fragment order
// ---------------------------------------------------------------------------
__device__ void stage_token_block(const __nv_bfloat16* __restrict__ xrow, int d,
                                  __half* __restrict__ x16row, float* __restrict__ xinv,
                                  float* red /* smem [32] */) {
    float amax = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) amax = fmaxf(amax, fabsf(__bfloat162float(xrow[i])));
    amax = warp_max(amax);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
        red[31] = m;
    }
    __syncthreads();
    const float mult = f16_range_mult(red[31]);
    if (threadIdx.x == 0) *xinv = 1.0f / mult;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        int tile = i >> 7;
        x16row[tile * 128 + kperm_pos(i & 127)] = __float2half_rn(__bfloat162float(xrow[i]) * mult);
    }
}

__device__ void stage_token_warp(const __nv_bfloat16* __restrict__ xrow, int d,
                                 __half* __restrict__ x16row, float* __restrict__ xinv) {
    const int lane = threadIdx.x & 31;
    float amax = 0.f;
    for (int i = lane; i < d; i += 32) amax = fmaxf(amax, fabsf(__bfloat162float(xrow[i])));
    amax = warp_max(amax);
    const float mult = f16_range_mult(amax);
    if (lane == 0) *xinv = 1.0f / mult;
    for (int i = lane; i < d; i += 32) {
        int tile = i >> 7;
        x16row[tile * 128 + kperm_pos(i & 127)] = __float2half_rn(__bfloat162float(xrow[i]) * mult);
    }
}

// ---------------------------------------------------------------------------
// a3: stable bucketing of a chunk of assignments by one CTA of 256 threads.
// Entries [a0, a1) are processed in rounds of 256 (8 warps x 32); within a
// round, ranks come from warp match + a per-warp count table.
// base[e] (smem) holds the first output position of expert e for this chunk
// and is advanced as entries are placed.
// ---------------------------------------------------------------------------
__device__ void bucket_place_block(const int* __restrict__ sel, int a0, int a1, int E,
                                   int* base /* smem [E] */, int* wcnt /* smem [8][E] */,
                                   int* __restrict__ perm, int* __restrict__ inv,
                                   uint32_t* status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r0 = a0; r0 < a1; r0 += kRouterThreads) {
        for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
        __syncthreads();
        const int a = r0 + threadIdx.x;
        int e = -1;
        if (a < a1) {
            e = sel[a];
            if (e < 0 || e >= E) {
                if (status) atomicOr(status, kStatusBadIndex);
                e = -1;
            }
        }
        const uint32_t m = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(m & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(m);
        __syncthreads();
        // exclusive scan over warps for every expert
        for (int x = threadIdx.x; x < E; x += blockDim.x) {
            int run = base[x];
            for (int w = 0; w < 8; ++w) {
                int c = wcnt[w * E + x];
                wcnt[w * E + x] = run;
                run += c;
            }
            base[x] = run;
        }
        __syncthreads();
        if (e >= 0) {
            int pos = wcnt[warp * E + e] + rank;
            perm[pos] = a;
            if (inv) inv[a] = pos;
        }
        __syncthreads();
    }
}

// Per-expert counts of a chunk into smem cnt[E] (zeroed by the caller).
__device__ void bucket_count_block(const int* __restrict__ sel, int a0, int a1, int E, int* cnt) {
    for (int a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
        int e = sel[a];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
}

// Offsets, active-slot list and metadata from total counts (one CTA).
__device__ void bucket_finish_block(const int* cnt /* smem [E] */, int E, int T, int k, int n_shared,
                                    int* offs_smem /* smem [E+1] */, int* __restrict__ offsets,
                                    int* __restrict__ slot_expert, int* __restrict__ slot_off,
                                    int* __restrict__ slot_cnt, int* __restrict__ meta) {
    if (threadIdx.x == 0) {
        int run = 0, ns = 0;
        for (int e = 0; e < E; ++e) {
            offs_smem[e] = run;
            if (cnt[e] > 0) {
                slot_expert[ns] = e;
                slot_off[ns] = run;
                slot_cnt[ns] = cnt[e];
                ++ns;
            }
            run += cnt[e];
        }
        offs_smem[E] = run;
        if (n_shared) {
            slot_expert[ns] = E;
            slot_off[ns] = T * k;
            slot_cnt[ns] = T;
            ++ns;
        }
        meta[0] = ns;
        meta[1] = T;
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = offs_smem[e];
}

struct RouterArgs {
    const __nv_bfloat16* x;
    const float* wr;
    const float* bias;
    int T, d, E, k, n_shared;
    Workspace ws;
};

// ---------------------------------------------------------------------------
// Fused decode router (T <= 64): logits, fp16 staging, and -- in the last CTA
// to finish -- top-k, renormalised weights and bucketing.
// grid = E/2 CTAs; warp w computes a quarter of the dot products of expert
// 2*blockIdx + w/4.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouterThreads) router_small_kernel(RouterArgs a) {
    __shared__ float part[8][kSmallT];
    __shared__ float red[32];
    __shared__ int s_cnt[256];
    __shared__ int s_offs[257];
    __shared__ int s_wcnt[8 * 256];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 2 + (warp >> 2);
    const int q = warp & 3;
    const int T = a.T, d = a.d;
    const int n_it = d >> 7;   // 128-element chunks of the row

    // router row chunks it = q, q+4, ... of expert e, 4 floats per lane
    float4 wv[kMaxKIt / 4 * 4 / 4 > 0 ? kMaxKIt : 1];
    int cnt_it = 0;
#pragma unroll
    for (int j = 0; j < kMaxKIt; ++j) {
        int it = q + 4 * j;
        if (it < n_it) {
            wv[j] = *reinterpret_cast<const float4*>(a.wr + (size_t)e * d + it * 128 + lane * 4);
            ++cnt_it;
        }
    }
    for (int t = 0; t < T; ++t) {
        float acc = 0.f;
        const __nv_bfloat16* xr = a.x + (size_t)t * d;
#pragma unroll
        for (int j = 0; j < kMaxKIt; ++j) {
            if (j < cnt_it) {
                int it = q + 4 * j;
                uint2 raw = *reinterpret_cast<const uint2*>(xr + it * 128 + lane * 4);
                __nv_bfloat162 p0 = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
                __nv_bfloat162 p1 = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
                acc = fmaf(wv[j].x, __low2float(p0), acc);
                acc = fmaf(wv[j].y, __high2float(p0), acc);
                acc = fmaf(wv[j].z, __low2float(p1), acc);
                acc = fmaf(wv[j].w, __high2float(p1), acc);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) part[warp][t] = acc;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * T; i += blockDim.x) {
        int ee = i / T, t = i % T;
        int ex = blockIdx.x * 2 + ee;
        float l = ((part[ee * 4 + 0][t] + part[ee * 4 + 1][t]) + part[ee * 4 + 2][t]) + part[ee * 4 + 3][t];
        l += a.bias[ex];
        a.ws.logits[(size_t)t * a.E + ex] = l;
    }
    // fp16 staging of token rows owned by this CTA
    for (int t = blockIdx.x; t < T; t += gridDim.x)
        stage_token_block(a.x + (size_t)t * d, d, a.ws.x16 + (size_t)t * d, a.ws.xinv + t, red);

    // last CTA to arrive finishes the routing
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t prev = atomicAdd(&a.ws.counters[0], 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // top-k per token: warp per token (logits read through L2)
    for (int t = warp; t < T; t += 8) {
        topk_warp<true>(a.ws.logits + (size_t)t * a.E, a.E, a.k, a.ws.idx + t * a.k, a.ws.w + t * a.k,
                        a.ws.status);
    }
    __syncthreads();
    __threadfence_block();
    // bucketing of the T*k assignments
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();
    const int n = T * a.k;
    bucket_count_block(a.ws.idx, 0, n, a.E, s_cnt);
    __syncthreads();
    bucket_finish_block(s_cnt, a.E, T, a.k, a.n_shared, s_offs, a.ws.offsets, a.ws.slot_expert,
                        a.ws.slot_off, a.ws.slot_cnt, a.ws.meta);
    __syncthreads();
    bucket_place_block(a.ws.idx, 0, n, a.E, s_offs, s_wcnt, a.ws.perm, a.ws.inv, a.ws.status);
    // reset per-position h maxima for the expert kernels
    const int P = T * (a.k + a.n_shared);
    for (int i = threadIdx.x; i < P; i += blockDim.x) a.ws.hamax[i] = 0u;
    if (threadIdx.x == 0) a.ws.counters[0] = 0u;
}

// ---------------------------------------------------------------------------
// Large-T router: tiled fp32 logits, then per-token top-k + staging, then a
// three-pass bucketing.
// ---------------------------------------------------------------------------
constexpr int kLTok = 64, kLExp = 64, kLK = 32;

__global__ void __launch_bounds__(256) router_logits_tiled(RouterArgs a) {
    __shared__ float xs[kLK][kLTok + 1];
    __shared__ float ws_[kLK][kLExp + 1];
    const int t0 = blockIdx.x * kLTok, e0 = blockIdx.y * kLExp;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 16 x 16 threads, 4 x 4 outputs each
    float acc[4][4] = {};
    for (int k0 = 0; k0 < a.d; k0 += kLK) {
        for (int i = threadIdx.x; i < kLTok * kLK; i += 256) {
            int tt = i / kLK, kk = i % kLK;
            int t = t0 + tt;
            xs[kk][tt] = (t < a.T) ? __bfloat162float(a.x[(size_t)t * a.d + k0 + kk]) : 0.f;
            int e = e0 + tt;
            ws_[kk][tt] = (e < a.E) ? a.wr[(size_t)e * a.d + k0 + kk] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kLK; ++kk) {
            float xv[4], wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[i] = xs[kk][ty * 4 + i];
                wv[i] = ws_[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int t = t0 + ty * 4 + i;
        if (t >= a.T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int e = e0 + tx * 4 + j;
            if (e < a.E) a.ws.logits[(size_t)t * a.E + e] = acc[i][j] + a.bias[e];
        }
    }
}

__global__ void __launch_bounds__(256) token_prep_kernel(RouterArgs a) {
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + warp;
    if (t >= a.T) return;
    topk_warp<false>(a.ws.logits + (size_t)t * a.E, a.E, a.k, a.ws.idx + t * a.k, a.ws.w + t * a.k,
                     a.ws.status);
    stage_token_warp(a.x + (size_t)t * a.d, a.d, a.ws.x16 + (size_t)t * a.d, a.ws.xinv + t);
}

struct BucketArgs {
    const int* sel;
    int n, T, E, k, n_shared;
    Workspace ws;
};

__global__ void __launch_bounds__(256) bucket_hist_kernel(BucketArgs a) {
    __shared__ int cnt[256];
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int a0 = blockIdx.x * kBucketChunk;
    const int a1 = min(a.n, a0 + kBucketChunk);
    bucket_count_block(a.sel, a0, a1, a.E, cnt);
    __syncthreads();
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) a.ws.chunk_hist[blockIdx.x * a.E + i] = cnt[i];
}

__global__ void __launch_bounds__(256) bucket_scan_kernel(BucketArgs a, int n_chunks) {
    __shared__ int cnt[256];
    __shared__ int offs[257];
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        int s = 0;
        for (int c = 0; c < n_chunks; ++c) s += a.ws.chunk_hist[c * a.E + e];
        cnt[e] = s;
    }
    __syncthreads();
    bucket_finish_block(cnt, a.E, a.T, a.k, a.n_shared, offs, a.ws.offsets, a.ws.slot_expert,
                        a.ws.slot_off, a.ws.slot_cnt, a.ws.meta);
    __syncthreads();
    // chunk bases: first output position of each (chunk, expert)
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        int run = offs[e];
        for (int c = 0; c < n_chunks; ++c) {
            int h = a.ws.chunk_hist[c * a.E + e];
            a.ws.chunk_hist[c * a.E + e] = run;
            run += h;
        }
    }
    const int P = a.T * (a.k + a.n_shared);
    for (int i = threadIdx.x; i < P; i += blockDim.x) a.ws.hamax[i] = 0u;
}

__global__ void __launch_bounds__(256) bucket_place_kernel(BucketArgs a) {
    __shared__ int base[256];
    __shared__ int wcnt[8 * 256];
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) base[i] = a.ws.chunk_hist[blockIdx.x * a.E + i];
    __syncthreads();
    const int a0 = blockIdx.x * kBucketChunk;
    const int a1 = min(a.n, a0 + kBucketChunk);
    bucket_place_block(a.sel, a0, a1, a.E, base, wcnt, a.ws.perm, a.ws.inv, a.ws.status);
}

__global__ void __launch_bounds__(256) topk_only_kernel(const float* logits, int T, int E, int k,
                                                        int* idx, float* w) {
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    topk_warp<false>(logits + (size_t)t * E, E, k, idx + t * k, w ? w + t * k : nullptr, nullptr);
}

RouterArgs make_args(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                     const Workspace& ws) {
    RouterArgs a;
    a.x = x;
    a.wr = L.router;
    a.bias = L.bias;
    a.T = T;
    a.d = s.d;
    a.E = s.E;
    a.k = s.k;
    a.n_shared = s.n_shared;
    a.ws = ws;
    return a;
}

}  // namespace

cudaError_t launch_bucket(const Shape& s, const int* idx, int T, const Workspace& ws,
                          cudaStream_t st, int* n_launch) {
    BucketArgs b;
    b.sel = idx;
    b.n = T * s.k;
    b.T = T;
    b.E = s.E;
    b.k = s.k;
    b.n_shared = s.n_shared;
    b.ws = ws;
    const int n_chunks = (b.n + kBucketChunk - 1) / kBucketChunk;
    bucket_hist_kernel<<<n_chunks, 256, 0, st>>>(b);
    bucket_scan_kernel<<<1, 256, 0, st>>>(b, n_chunks);
    bucket_place_kernel<<<n_chunks, 256, 0, st>>>(b);
    *n_launch += 3;
    return cudaGetLastError();
}

cudaError_t launch_router(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                          const Workspace& ws, cudaStream_t st, int* n_launch) {
    RouterArgs a = make_args(s, L, x, T, ws);
    if (T <= kSmallT) {
        router_small_kernel<<<s.E / 2, kRouterThreads, 0, st>>>(a);
        *n_launch += 1;
        return cudaGetLastError();
    }
    dim3 g1((T + kLTok - 1) / kLTok, (s.E + kLExp - 1) / kLExp);
    router_logits_tiled<<<g1, 256, 0, st>>>(a);
    token_prep_kernel<<<(T + 7) / 8, 256, 0, st>>>(a);
    *n_launch += 2;
    return launch_bucket(s, ws.idx, T, ws, st, n_launch);
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int* idx, float* w,
                        cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    topk_only_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, T, E, k, idx, w);
    return cudaGetLastError();
}

}  // namespace flint
