// One decode step of Flint-shaped attention: per sequence one new token, 32
// query heads sharing 4 key-value heads in groups of 8, head dimension 128,
// per-head QK RMSNorm, rotary positions on sliding-window layers, learned
// per-head sinks, a 513-token window (the current token and the 512 before
// it) or full attention ("Recursive Flint 40B-A2.5B", section "The
// architecture is an argument about memory bandwidth", Attention and
// Position-encoding bullets).
//
// One CTA per (sequence, key-value head), one warp per query head of the
// group. The window's keys and values (bf16 cache rows) stream through
// shared memory in tiles of 64 positions with 16-byte asynchronous copies,
// two tiles in flight; each warp keeps an online softmax (running max, sum
// and the 128-wide output accumulator, four dimensions per lane) in fp32.
// The current token's key and value enter unrounded and are then stored,
// bf16, in its cache slot.
#include "../../include/flint_moe.h"
#include "kernels.cuh"

namespace flint {

namespace {

constexpr int kAD = 128;                 // head dimension
constexpr int kAGroup = 8;               // query heads per key-value head (= warps)
constexpr int kATile = 64;               // positions per shared-memory tile
constexpr int kARow = kAD * 2 + 16;      // bytes per cached row in shared memory (padded: conflict-free rows)
constexpr int kATileBytes = kATile * kARow;

struct AttnArgs {
    const __nv_bfloat16* q;    // [B][H][128]
    const __nv_bfloat16* k;    // [B][KV][128]
    const __nv_bfloat16* v;    // [B][KV][128]
    __nv_bfloat16* kc;         // [B][KV][cap][128]
    __nv_bfloat16* vc;
    const int32_t* pos;        // [B]
    const float* wq;           // [128]
    const float* wk;           // [128]
    const float* sinks;        // [H]
    __nv_bfloat16* out;        // [B][H][128]
    int H, KV, window, cap, rope;
    double log2_theta;
    float eps;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// RMSNorm and (optionally) the rotation of one head held as four dimensions
// per lane: lane l has dims l, l+32, l+64, l+96, so the rotated pairs
// (i, i+64) are (v0, v2) and (v1, v3).
__device__ __forceinline__ void norm_rope(float (&v)[4], const float* w, int lane, int pos, const AttnArgs& a) {
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    ss = warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss / (float)kAD + a.eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = v[i] * inv * __ldg(w + lane + 32 * i);
    if (a.rope) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = lane + 32 * j;   // pair index
            // the angle in double and reduced modulo 2 pi, so that large
            // positions keep full precision
            const double f = exp2(-(double)i / 64.0 * a.log2_theta);
            double ang = (double)pos * f;
            ang -= 6.283185307179586476925 * floor(ang / 6.283185307179586476925);
            float sn, cs;
            sincosf((float)ang, &sn, &cs);
            const float x0 = v[j], x1 = v[j + 2];
            v[j] = x0 * cs - x1 * sn;
            v[j + 2] = x0 * sn + x1 * cs;
        }
    }
}

constexpr int kASmem = 4 * kATileBytes;   // two buffers of key rows, two of value rows

__global__ void __launch_bounds__(256) attn_decode_kernel(AttnArgs a) {
    extern __shared__ __align__(16) uint8_t asmem[];
    uint8_t* ks[2] = {asmem, asmem + kATileBytes};
    uint8_t* vs[2] = {asmem + 2 * kATileBytes, asmem + 3 * kATileBytes};
    __shared__ __align__(16) float qs[kAGroup][kAD];
    __shared__ __align__(16) float kcur[kAD], vcur[kAD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x, b = blockIdx.y;
    const int h = g * kAGroup + warp;
    const int pos = a.pos[b];
    const int n_prev = a.window > 0 ? min(pos, a.window - 1) : pos;
    const int first = pos - n_prev;
    const size_t cache_base = ((size_t)b * a.KV + g) * a.cap;
    const __nv_bfloat16* kcg = a.kc + cache_base * kAD;
    const __nv_bfloat16* vcg = a.vc + cache_base * kAD;
    const int n_tiles = (n_prev + kATile - 1) / kATile;

    // request the first two tiles of cached rows before anything else
    auto load_tile = [&](int tile, int buf) {
        const int p0 = first + tile * kATile;
        for (int i = threadIdx.x; i < kATile * 16; i += blockDim.x) {
            const int r = i >> 4, c = i & 15;
            if (p0 + r < pos) {
                const size_t slot = (size_t)((p0 + r) % a.cap);
                cp_async16(ks[buf] + r * kARow + c * 16, kcg + slot * kAD + c * 8);
                cp_async16(vs[buf] + r * kARow + c * 16, vcg + slot * kAD + c * 8);
            }
        }
        cp_async_commit();
    };
    if (n_tiles > 0) load_tile(0, 0);
    if (n_tiles > 1) load_tile(1, 1);

    // this warp's query head, and (warp 0) the current key and value
    float q[4];
    {
        const __nv_bfloat16* qr = a.q + ((size_t)b * a.H + h) * kAD;
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = __bfloat162float(qr[lane + 32 * i]);
        norm_rope(q, a.wq, lane, pos, a);
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[warp][lane + 32 * i] = q[i];
    }
    if (warp == 0) {
        float kv[4];
        const __nv_bfloat16* kr = a.k + ((size_t)b * a.KV + g) * kAD;
        const __nv_bfloat16* vr = a.v + ((size_t)b * a.KV + g) * kAD;
#pragma unroll
        for (int i = 0; i < 4; ++i) kv[i] = __bfloat162float(kr[lane + 32 * i]);
        norm_rope(kv, a.wk, lane, pos, a);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            kcur[lane + 32 * i] = kv[i];
            vcur[lane + 32 * i] = __bfloat162float(vr[lane + 32 * i]);
        }
    }
    __syncthreads();

    const float scale = rsqrtf((float)kAD);   // 1/sqrt(128), exact: 2^-3.5 rounded once
    float m = -INFINITY, l = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const float4* q4 = reinterpret_cast<const float4*>(qs[warp]);
    for (int tile = 0; tile < n_tiles; ++tile) {
        const int buf = tile & 1;
        if (tile + 1 < n_tiles) cp_async_wait<1>(); else cp_async_wait<0>();
        __syncthreads();
        const int p0 = first + tile * kATile;
        const int nk = min(kATile, pos - p0);
        // scores of keys lane and lane + 32
        float s[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = lane + 32 * j;
            float dot = 0.f;
            if (r < nk) {
                const uint4* kr = reinterpret_cast<const uint4*>(ks[buf] + r * kARow);
#pragma unroll 4
                for (int c = 0; c < 16; ++c) {
                    const uint4 kw = kr[c];
                    const float4 qa = q4[2 * c], qb = q4[2 * c + 1];
                    const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kw);
                    const float2 k01 = __bfloat1622float2(k2[0]), k23 = __bfloat1622float2(k2[1]);
                    const float2 k45 = __bfloat1622float2(k2[2]), k67 = __bfloat1622float2(k2[3]);
                    dot = fmaf(qa.x, k01.x, dot);
                    dot = fmaf(qa.y, k01.y, dot);
                    dot = fmaf(qa.z, k23.x, dot);
                    dot = fmaf(qa.w, k23.y, dot);
                    dot = fmaf(qb.x, k45.x, dot);
                    dot = fmaf(qb.y, k45.y, dot);
                    dot = fmaf(qb.z, k67.x, dot);
                    dot = fmaf(qb.w, k67.y, dot);
                }
                s[j] = dot * scale;
            } else {
                s[j] = -INFINITY;
            }
        }
        const float tmax = warp_max(fmaxf(s[0], s[1]));
        const float m_new = fmaxf(m, tmax);
        const float corr = expf(m - m_new);   // 0 on the first tile (m = -inf)
        float p[2];
        p[0] = expf(s[0] - m_new);
        p[1] = expf(s[1] - m_new);
        l = l * corr + warp_sum(p[0] + p[1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] *= corr;
        m = m_new;
        // acc[d] += sum_r p_r V[r][d]
        for (int r = 0; r < nk; ++r) {
            const float pr = __shfl_sync(0xffffffffu, p[r >> 5], r & 31);
            const __nv_bfloat16* vrow = reinterpret_cast<const __nv_bfloat16*>(vs[buf] + r * kARow);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(pr, __bfloat162float(vrow[lane + 32 * i]), acc[i]);
        }
        __syncthreads();   // every warp is done with this buffer
        if (tile + 2 < n_tiles) load_tile(tile + 2, buf);
    }
    // the current token, unrounded
    {
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) dot = fmaf(q[i], kcur[lane + 32 * i], dot);
        const float sc = warp_sum(dot) * scale;
        const float m_new = fmaxf(m, sc);
        const float corr = expf(m - m_new);
        const float pc = expf(sc - m_new);
        l = l * corr + pc;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = acc[i] * corr + pc * vcur[lane + 32 * i];
        m = m_new;
    }
    // the sink joins the denominator only
    {
        const float sk = __ldg(a.sinks + h);
        const float m_new = fmaxf(m, sk);
        const float corr = expf(m - m_new);
        l = l * corr + expf(sk - m_new);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] *= corr;
    }
    const float inv = 1.0f / l;
    __nv_bfloat16* o = a.out + ((size_t)b * a.H + h) * kAD;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
    // store the current key and value, bf16, in the position's slot (outside
    // the window that was read: cap >= window)
    if (warp == 0) {
        const size_t slot = (size_t)(pos % a.cap);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a.kc[(cache_base + slot) * kAD + lane + 32 * i] = __float2bfloat16_rn(kcur[lane + 32 * i]);
            a.vc[(cache_base + slot) * kAD + lane + 32 * i] = __float2bfloat16_rn(vcur[lane + 32 * i]);
        }
    }
}

}  // namespace

}  // namespace flint

extern "C" flint_status flint_moe_attn_decode(const flint_moe_attn_config* cfg, int B, const void* q_dev, const void* k_dev,
                                          const void* v_dev, void* k_cache_dev, void* v_cache_dev,
                                          const int32_t* pos_dev, const float* q_norm_w_dev,
                                          const float* k_norm_w_dev, const float* sinks_dev, void* out_dev,
                                          void* stream) {
    using namespace flint;
    if (cfg == nullptr || B < 0) return FLINT_EINVAL;
    if (cfg->head_dim != kAD || cfg->n_kv < 1 || cfg->n_kv > 64 || cfg->n_heads != cfg->n_kv * kAGroup)
        return FLINT_EINVAL;
    if (cfg->window < 0 || cfg->cap < 1 || (cfg->window > 0 && cfg->cap < cfg->window)) return FLINT_EINVAL;
    if (!(cfg->rope_theta > 1.0f) || !(cfg->eps >= 0.0f) || (cfg->rope != 0 && cfg->rope != 1)) return FLINT_EINVAL;
    if (B == 0) return FLINT_OK;
    const void* ptrs[] = {q_dev, k_dev, v_dev, k_cache_dev, v_cache_dev, pos_dev, q_norm_w_dev, k_norm_w_dev,
                          sinks_dev, out_dev};
    for (const void* p : ptrs)
        if (p == nullptr) return FLINT_EINVAL;
    if (((uintptr_t)k_cache_dev & 15u) || ((uintptr_t)v_cache_dev & 15u)) return FLINT_EINVAL;
    AttnArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q_dev);
    a.k = static_cast<const __nv_bfloat16*>(k_dev);
    a.v = static_cast<const __nv_bfloat16*>(v_dev);
    a.kc = static_cast<__nv_bfloat16*>(k_cache_dev);
    a.vc = static_cast<__nv_bfloat16*>(v_cache_dev);
    a.pos = pos_dev;
    a.wq = q_norm_w_dev;
    a.wk = k_norm_w_dev;
    a.sinks = sinks_dev;
    a.out = static_cast<__nv_bfloat16*>(out_dev);
    a.H = cfg->n_heads;
    a.KV = cfg->n_kv;
    a.window = cfg->window;
    a.cap = cfg->cap;
    a.rope = cfg->rope;
    a.log2_theta = log2((double)cfg->rope_theta);
    a.eps = cfg->eps;
    static bool opted_in = false;   // the attribute is per device function, set once
    if (!opted_in) {
        if (cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kASmem) !=
            cudaSuccess) {
            cudaGetLastError();
            return FLINT_ECUDA;
        }
        opted_in = true;
    }
    attn_decode_kernel<<<dim3(cfg->n_kv, B), 256, kASmem, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? FLINT_OK : FLINT_ECUDA;
}
