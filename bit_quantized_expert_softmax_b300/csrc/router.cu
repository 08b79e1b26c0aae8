// Router (logits, top-k, renormalised softmax), fp16 staging of the hidden
// states, and token -> expert bucketing.
//
// Structure from the Flint blog ("Recursive Flint 40B-A2.5B", section "The
// architecture is an argument about memory bandwidth", Sparsity bullet): 256
// routed experts, 6 chosen per token, one always-on shared expert. The
// routing rule: fp32 logits, the k largest (ties: lower expert index),
// softmax renormalised over the chosen k.
#include <float.h>

#include <algorithm>

#include "kernels.cuh"
#include "pdl.cuh"
#include "topk.cuh"

namespace flint {

namespace {

constexpr int kRouterThreads = 256;   // 8 warps

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
            e = __ldcg(sel + a);   // written earlier in this kernel or the previous one
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
        const int e = __ldcg(sel + a);
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
}

// Exclusive prefix sum of one int per thread over a block of 256 threads;
// *total receives the sum of all. wsum: shared scratch of 8 ints.
__device__ __forceinline__ int block_exclusive_scan_256(int v, int* wsum, int* total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < 8 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < 8) wsum[lane] = w;
    }
    __syncthreads();
    const int base = warp > 0 ? wsum[warp - 1] : 0;
    *total = wsum[7];
    __syncthreads();
    return base + x - v;
}

// Offsets, active-slot list and metadata from total counts, by one CTA of 256
// threads (thread e owns expert e): one block scan over (count | nonempty<<20)
// gives both the offset and the active-slot index of every expert.
__device__ void bucket_finish_block(const int* cnt /* smem [E] */, int E, int T, int k, int n_shared,
                                    int* offs_smem /* smem [E+1] */, int* __restrict__ offsets,
                                    int* __restrict__ slot_expert, int* __restrict__ slot_off,
                                    int* __restrict__ slot_cnt, int* __restrict__ meta) {
    __shared__ int wsum[8];
    const int e = threadIdx.x;
    const int c = e < E ? cnt[e] : 0;
    const int packed = c | ((c > 0 ? 1 : 0) << 20);
    int total = 0;
    const int excl = block_exclusive_scan_256(packed, wsum, &total);
    const int off = excl & 0xfffff, slot = excl >> 20;
    if (e < E) {
        offs_smem[e] = off;
        offsets[e] = off;
        if (c > 0) {
            slot_expert[slot] = e;
            slot_off[slot] = off;
            slot_cnt[slot] = c;
        }
    }
    if (threadIdx.x == 0) {
        const int n_assign = total & 0xfffff;
        int ns = total >> 20;
        offs_smem[E] = n_assign;
        offsets[E] = n_assign;
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
}

struct RouterArgs {
    const __nv_bfloat16* x;
    const float* wr;
    const float* bias;
    int T, d, E, k, n_shared;
    int stage_x16;   // large-T path: also stage fp16 hidden states for the mma.sync experts
    Workspace ws;
};

// ---------------------------------------------------------------------------
// Fused decode router (T <= 64): logits, fp16 staging, and -- in the last CTA
// to finish -- top-k, renormalised weights and bucketing.
//
// grid = (E/8 expert groups, ceil(T/16) token groups). A CTA bulk-copies its 8
// fp32 router rows and its (up to) 16 bf16 hidden rows into shared memory and
// forms the 16 x 8 logit tile on the tensor cores (mma.sync m16n8k16, bf16
// operands, fp32 accumulation): the hidden states are bf16 and exact as the A
// operand; each fp32 router weight is split in registers into
// hi = bf16(w) and lo = bf16(w - hi), and the two products are accumulated,
// which keeps ~16 significant bits of w (relative error of a logit ~2^-16,
// inside the router's 1e-4 tolerance). Warp w takes the 16-element K steps
// w, w + 8, ...; the 8 partial tiles are summed in a fixed order.
// ---------------------------------------------------------------------------
constexpr int kTokGroup = 16;   // tokens per CTA: the M of the tile
constexpr int kRouterExp = 8;   // experts per CTA: the N of the tile
// the fragment loads read 16 hidden rows and the partial tiles hold 16 x 8
// values: the staging buffer and the tile must have exactly these sizes
static_assert(kTokGroup == 16 && kRouterExp == 8, "one m16n8 tile per CTA");
// arrival counters of the token groups of router_small_kernel (after the
// ones the expert kernels use)
constexpr int kGroupCounters = kCounters - kSmallT / kTokGroup;
static_assert(kGroupCounters > 64, "counter ranges overlap");

// Shared-memory row pitches: 32 bytes past a router row and 16 past a hidden
// row, so that the fragment loads of 8 rows hit distinct banks.
__host__ __device__ __forceinline__ size_t rs_wpitch(int d) { return (size_t)d * 4 + 32; }
__host__ __device__ __forceinline__ size_t rs_xpitch(int d) { return (size_t)d * 2 + 16; }

// bf16 x bf16 -> fp32 m16n8k16 (A row-major 16 x 16, B "col" 16 x 8)
__device__ __forceinline__ void rmma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// two fp32 weights (consecutive K) -> their bf16 hi pair and lo pair
__device__ __forceinline__ void split_pair(float2 w, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(w.x, w.y);
    const __nv_bfloat162 l = __floats2bfloat162_rn(w.x - __low2float(h), w.y - __high2float(h));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

__global__ void __launch_bounds__(kRouterThreads) router_small_kernel(RouterArgs a) {
    griddep_wait();
    // [8][d] fp32 router rows, then [16][d] bf16 hidden rows (padded pitches);
    // the bucketing CTA reuses the buffer for its tables once its logits are
    // done
    extern __shared__ __align__(128) uint8_t rsm[];
    __shared__ uint64_t rbar;
    __shared__ float red[32];
    __shared__ float part[8][kTokGroup * kRouterExp];
    __shared__ int s_last;
    int* s_wcnt = reinterpret_cast<int*>(rsm);   // [8][256]
    int* s_cnt = s_wcnt + 8 * 256;               // [256]
    int* s_offs = s_cnt + 256;                   // [257]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, d = a.d;
    const int e0 = blockIdx.x * kRouterExp;
    const int t0 = blockIdx.y * kTokGroup;
    const int nt = min(kTokGroup, T - t0);
    const size_t wp = rs_wpitch(d), xp = rs_xpitch(d);
    uint8_t* wsm = rsm;
    uint8_t* xsm = rsm + kRouterExp * wp;
    if (threadIdx.x == 0) {
        mbar_init(&rbar, 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(&rbar, (uint32_t)(kRouterExp * d * 4 + nt * d * 2));
        for (int j = 0; j < kRouterExp; ++j)
            bulk_g2s(wsm + j * wp, a.wr + (size_t)(e0 + j) * d, (uint32_t)(d * 4), &rbar);
        for (int r = 0; r < nt; ++r) bulk_g2s(xsm + r * xp, a.x + (size_t)(t0 + r) * d, (uint32_t)(d * 2), &rbar);
    }
    // rows of absent tokens are zero (their logits are not stored)
    for (int r = nt; r < kTokGroup; ++r)
        for (int i = threadIdx.x; i < d / 8; i += blockDim.x)
            *reinterpret_cast<uint4*>(xsm + r * xp + i * 16) = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const bool w_ok = mbar_wait_bounded(&rbar, 0, a.ws.status);
    const bool ok = __syncthreads_and(w_ok ? 1 : 0) != 0;
    if (ok) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        // A (ldmatrix x4): lanes 0-7 rows 0-7 / 8-15 rows 8-15 at K 0..7,
        // lanes 16-31 the same rows at K 8..15
        const uint8_t* arow = xsm + ((lane & 7) + 8 * ((lane >> 3) & 1)) * xp + 16 * (lane >> 4);
        // B: expert lane/4, K pair 2 (lane % 4) and that pair + 8
        const float* brow = reinterpret_cast<const float*>(wsm + (lane >> 2) * wp) + 2 * (lane & 3);
        for (int k0 = warp * 16; k0 < d; k0 += 8 * 16) {
            uint32_t af[4];
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(af[0]), "=r"(af[1]), "=r"(af[2]), "=r"(af[3])
                         : "r"(smem_u32(arow + k0 * 2)));
            uint32_t h0, l0, h1, l1;
            split_pair(*reinterpret_cast<const float2*>(brow + k0), h0, l0);
            split_pair(*reinterpret_cast<const float2*>(brow + k0 + 8), h1, l1);
            rmma_bf16(c, af, h0, h1);
            rmma_bf16(c, af, l0, l1);
        }
        // C: rows lane/4 (c0, c1) and lane/4 + 8 (c2, c3), columns 2 (lane % 4) + {0, 1}
        const int r = lane >> 2, col = 2 * (lane & 3);
        part[warp][r * kRouterExp + col] = c[0];
        part[warp][r * kRouterExp + col + 1] = c[1];
        part[warp][(r + 8) * kRouterExp + col] = c[2];
        part[warp][(r + 8) * kRouterExp + col + 1] = c[3];
    }
    __syncthreads();
    if (ok && threadIdx.x < kTokGroup * kRouterExp) {
        const int r = threadIdx.x / kRouterExp, col = threadIdx.x % kRouterExp;
        float s = part[0][threadIdx.x];
#pragma unroll
        for (int w = 1; w < 8; ++w) s += part[w][threadIdx.x];
        if (r < nt) a.ws.logits[(size_t)(t0 + r) * a.E + e0 + col] = s + a.bias[e0 + col];
    }
    // fp16 staging: CTA (p, g) stages tokens 16g + p, 16g + p + gridDim.x, ...
    // from its own copy of the hidden rows
    for (int p = blockIdx.x; p < nt; p += gridDim.x) {
        const int t = t0 + p;
        const __nv_bfloat16* xr = ok ? reinterpret_cast<const __nv_bfloat16*>(xsm + p * xp) : a.x + (size_t)t * d;
        stage_token_block(xr, d, a.ws.x16 + (size_t)t * d, a.ws.xinv + t, red);
    }

    // the last CTA of this token group takes the top-k of its tokens (a warp
    // per token, logits read through L2) ...
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(&a.ws.counters[kGroupCounters + blockIdx.y], 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int r = warp; r < nt; r += 8)
        topk_warp<true>(a.ws.logits + (size_t)(t0 + r) * a.E, a.E, a.k, a.ws.idx + (t0 + r) * a.k,
                        a.ws.w + (t0 + r) * a.k, a.ws.status);
    if (threadIdx.x == 0) a.ws.counters[kGroupCounters + blockIdx.y] = 0u;
    // ... and the last token group to finish buckets all of them
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(&a.ws.counters[0], 1u);
        s_last = (prev == gridDim.y - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
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
    griddep_wait();
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
    griddep_wait();
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + warp;
    if (t >= a.T) return;
    topk_warp<false>(a.ws.logits + (size_t)t * a.E, a.E, a.k, a.ws.idx + t * a.k, a.ws.w + t * a.k,
                     a.ws.status);
    if (a.stage_x16) stage_token_warp(a.x + (size_t)t * a.d, a.d, a.ws.x16 + (size_t)t * a.d, a.ws.xinv + t);
}

struct BucketArgs {
    const int* sel;
    int n, T, E, k, n_shared;
    int reset_hamax;   // clear the per-position h maxima the 16-bit-activation expert kernels accumulate
    Workspace ws;
};

__global__ void __launch_bounds__(256) bucket_hist_kernel(BucketArgs a) {
    griddep_wait();
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
    griddep_wait();
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
    if (a.reset_hamax) {
        const int P = a.T * (a.k + a.n_shared);
        for (int i = threadIdx.x; i < P; i += blockDim.x) a.ws.hamax[i] = 0u;
    }
}

__global__ void __launch_bounds__(256) bucket_place_kernel(BucketArgs a) {
    griddep_wait();
    __shared__ int base[256];
    __shared__ int wcnt[8 * 256];
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) base[i] = a.ws.chunk_hist[blockIdx.x * a.E + i];
    __syncthreads();
    const int a0 = blockIdx.x * kBucketChunk;
    const int a1 = min(a.n, a0 + kBucketChunk);
    bucket_place_block(a.sel, a0, a1, a.E, base, wcnt, a.ws.perm, a.ws.inv, a.ws.status);
}

// Routing of the FP4 prefill path: top-k and renormalised weights per token
// (a warp per token) and, for each of the token's k assignments, its rank
// within its expert, taken with one atomic per assignment into ws.ecount and
// left in ws.inv (the quantiser of x turns it into the bucketed position).
// The order of the rows inside an expert is free on that path -- every row is
// computed on its own and the combine reads rows by assignment -- so the
// atomics' arrival order changes no result.
// Top-k of 8 consecutive tokens per CTA (one per warp), then every
// assignment's rank within its expert: ranks inside the CTA from
// shared-memory counters, and one global atomic per (CTA, expert) for the
// CTA's base, so a popular expert's counter sees one atomic per CTA instead
// of one per assignment (four tokens per warp, one after the other, measured
// slower: the top-k chains are serial). Rows of one expert come out in an arbitrary
// order, which changes no result (every row is computed on its own and the
// combine finds it through inv).
constexpr int kRankTokPerWarp = 1;

__global__ void __launch_bounds__(256) token_rank_kernel(RouterArgs a) {
    griddep_wait();
    __shared__ int s_cnt[256];
    __shared__ int s_base[256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    int eid[kRankTokPerWarp], loc[kRankTokPerWarp];
#pragma unroll
    for (int i = 0; i < kRankTokPerWarp; ++i) {
        const int t = (blockIdx.x * 8 + warp) * kRankTokPerWarp + i;
        eid[i] = -1;
        loc[i] = 0;
        if (t < a.T) {
            const int e = topk_warp<false>(a.ws.logits + (size_t)t * a.E, a.E, a.k, a.ws.idx + t * a.k,
                                           a.ws.w + t * a.k, a.ws.status);
            if (lane < a.k) {
                if (e >= 0 && e < a.E) {
                    eid[i] = e;
                    loc[i] = atomicAdd(&s_cnt[e], 1);
                }
            }
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        const int n = s_cnt[e];
        s_base[e] = n > 0 ? atomicAdd(a.ws.ecount + e * kEcountStride, n) : 0;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRankTokPerWarp; ++i) {
        const int t = (blockIdx.x * 8 + warp) * kRankTokPerWarp + i;
        if (eid[i] >= 0) a.ws.inv[t * a.k + lane] = s_base[eid[i]] + loc[i];
    }
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
    a.stage_x16 = 1;
    a.ws = ws;
    return a;
}

}  // namespace

cudaError_t launch_bucket(const Shape& s, const int* idx, int T, const Workspace& ws,
                          cudaStream_t st, int* n_launch, bool reset_hamax) {
    BucketArgs b;
    b.reset_hamax = reset_hamax ? 1 : 0;
    b.sel = idx;
    b.n = T * s.k;
    b.T = T;
    b.E = s.E;
    b.k = s.k;
    b.n_shared = s.n_shared;
    b.ws = ws;
    const int n_chunks = (b.n + kBucketChunk - 1) / kBucketChunk;
    cudaError_t e = launch_pdl(bucket_hist_kernel, dim3(n_chunks), dim3(256), 0, st, b);
    if (e == cudaSuccess) e = launch_pdl(bucket_scan_kernel, dim3(1), dim3(256), 0, st, b, n_chunks);
    if (e == cudaSuccess) e = launch_pdl(bucket_place_kernel, dim3(n_chunks), dim3(256), 0, st, b);
    *n_launch += 3;
    return e;
}

// Dynamic shared memory the fused router may use (set once per device).
constexpr size_t kRouterDynSmemMax = 160 * 1024;

cudaError_t prepare_router() {
    const cudaError_t e = cudaFuncSetAttribute(router_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kRouterDynSmemMax);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

namespace {
// the router rows and hidden rows, or the bucketing tables if larger
size_t router_small_smem(const Shape& s) {
    return std::max((size_t)kRouterExp * rs_wpitch(s.d) + (size_t)kTokGroup * rs_xpitch(s.d),
                    (size_t)(8 * 256 + 256 + 257) * 4);
}
}  // namespace

bool router_fused(const Shape& s, int T) { return T <= kSmallT && router_small_smem(s) <= kRouterDynSmemMax; }

cudaError_t launch_router(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                          const Workspace& ws, cudaStream_t st, int* n_launch, bool stage_x16) {
    RouterArgs a = make_args(s, L, x, T, ws);
    a.stage_x16 = stage_x16 ? 1 : 0;
    const size_t smem = router_small_smem(s);
    if (router_fused(s, T)) {
        *n_launch += 1;
        return launch_pdl(router_small_kernel, dim3(s.E / kRouterExp, (T + kTokGroup - 1) / kTokGroup),
                          dim3(kRouterThreads), smem, st, a);
    }
    if (L.umma_router) {
        const cudaError_t e = launch_router_umma(s, L, x, T, ws.logits, ws.status, st);
        if (e != cudaSuccess) return e;
    } else {
        dim3 g1((T + kLTok - 1) / kLTok, (s.E + kLExp - 1) / kLExp);
        const cudaError_t e = launch_pdl(router_logits_tiled, g1, dim3(256), 0, st, a);
        if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_pdl(token_prep_kernel, dim3((T + 7) / 8), dim3(256), 0, st, a);
    if (e != cudaSuccess) return e;
    *n_launch += 2;
    // the FP4 expert path (no fp16 staging) does not use the h maxima
    return launch_bucket(s, ws.idx, T, ws, st, n_launch, stage_x16);
}

cudaError_t launch_router_fp4(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T, const Workspace& ws,
                              cudaStream_t st, int* n_launch) {
    RouterArgs a = make_args(s, L, x, T, ws);
    a.stage_x16 = 0;
    if (L.umma_router) {
        const cudaError_t e = launch_router_umma(s, L, x, T, ws.logits, ws.status, st);
        if (e != cudaSuccess) return e;
    } else {
        dim3 g1((T + kLTok - 1) / kLTok, (s.E + kLExp - 1) / kLExp);
        const cudaError_t el = launch_pdl(router_logits_tiled, g1, dim3(256), 0, st, a);
        if (el != cudaSuccess) return el;
    }
    const cudaError_t e = launch_pdl(token_rank_kernel, dim3((T + 8 * kRankTokPerWarp - 1) / (8 * kRankTokPerWarp)),
                                     dim3(256), 0, st, a);
    *n_launch += 2;
    return e;
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int* idx, float* w,
                        cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    topk_only_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, T, E, k, idx, w);
    return cudaGetLastError();
}

}  // namespace flint
