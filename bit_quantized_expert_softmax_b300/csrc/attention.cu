// One decode step of Flint-shaped attention: per sequence one new token, 32
// query heads sharing 4 key-value heads in groups of 8, head dimension 128,
// per-head QK RMSNorm, rotary positions on sliding-window layers, learned
// per-head sinks, a 513-token window (the current token and the 512 before
// it) or full attention ("Recursive Flint 40B-A2.5B", section "The
// architecture is an argument about memory bandwidth", Attention and
// Position-encoding bullets).
//
// One CTA per (sequence, key-value head), two per SM. The window's keys and
// values (bf16 cache rows) stream through shared memory in tiles of 64
// positions with 16-byte asynchronous copies, three tiles in flight. Both
// contractions of a tile run on the tensor cores (mma.sync, bf16 operands,
// fp32 accumulation), the group's 8 query heads as the MMA's N; the query and
// the probabilities enter as bf16 hi + lo pairs, so the scores and the
// weighted sum keep about 16 significant bits per operand. The softmax is
// online (running max and sum per head, in fp32). The current token's key and
// value enter unrounded and are then stored, bf16, in its cache slot.
#include <cmath>

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
    // rotary frequency of pair i as a fraction of a turn per position, in
    // 2^-64 turns: pos * rope_turns[i] (64-bit, wrapping) is the angle
    // modulo one turn, exactly up to the table's rounding
    unsigned long long rope_turns[kAD / 2];
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
            // the angle as a fraction of a turn: integer arithmetic keeps
            // large positions exact; the top 24 bits, in half-turns, go to
            // sincospif
            const unsigned long long turns = (unsigned long long)(unsigned)pos * a.rope_turns[i];
            // rounded to 24 bits (2^24 is a whole turn: sin and cos come out right)
            const float half_turns = (float)(unsigned)((turns + (1ull << 39)) >> 40) * 0x1p-23f;   // in [0, 2]
            float sn, cs;
            sincospif(half_turns, &sn, &cs);
            const float x0 = v[j], x1 = v[j + 2];
            v[j] = x0 * cs - x1 * sn;
            v[j + 2] = x0 * sn + x1 * cs;
        }
    }
}

// bf16 x bf16 -> fp32 m16n8k16 (A row-major 16 x 16, B "col" 16 x 8)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// v = hi + lo with hi = bf16(v), lo = bf16(v - hi): together ~16 significant bits
__device__ __forceinline__ void split_bf16x2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

constexpr int kAStages = 3;                                // tiles of key and value rows in flight
constexpr int kASmem = kAStages * 2 * kATileBytes;

// Shared scratch besides the tiles. The score and probability rows are
// padded so that the MMA fragments' stores and loads (lane (g, c) at row
// 2c / g, column g / c) fall in distinct banks.
constexpr int kAScRow = kATile + 4;
constexpr int kAPRow = kATile / 2 + 4;
struct AttnShared {
    union {
        float qs[kAGroup][kAD];       // normed (rotated) query heads, fp32 (before the tile loop)
        float sc[2][kAGroup][kAScRow]; // scores of the tile: the q_hi and q_lo parts, [head][key]
    };
    float kcur[kAD], vcur[kAD];       // the current token's key (normed, rotated) and value
    uint32_t ph[kAGroup][kAPRow];     // probabilities of the tile, bf16 hi parts, [head][key pair]
    uint32_t pl[kAGroup][kAPRow];     // and lo parts
    float corr[kAGroup];              // per head: rescale of the accumulators for this tile
    float fin_a[kAGroup], fin_b[kAGroup], fin_inv[kAGroup];   // the final current-token / sink fold
};

// One CTA per (key-value head g, sequence b); warp w is query head 8 g + w
// for the softmax and owns output dimensions 16 w .. 16 w + 15 for P.V.
// Per tile of 64 cached positions:
//   scores  S[key][head] = K[key][:] . Q[head][:] on the tensor cores, keys as
//           M (four 16-key m-tiles), the group's 8 heads as N, Q split into
//           bf16 hi + lo (warps 0-3: hi, 4-7: lo; one m-tile each)
//   softmax warp h: running max, rescale factor, p = exp(s - max), row sum
//   P.V     O^T[dim][head] += V^T[dim][key] . P^T[key][head], V^T by
//           transposing loads of the value rows, P split into hi + lo
// so both contractions keep about fp32 accuracy.
__global__ void __launch_bounds__(256, 2) attn_decode_kernel(AttnArgs a) {
    extern __shared__ __align__(16) uint8_t asmem[];
    __shared__ __align__(16) AttnShared sh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int g = blockIdx.x, b = blockIdx.y;
    const int h = g * kAGroup + warp;
    const int pos = a.pos[b];
    const int n_prev = a.window > 0 ? min(pos, a.window - 1) : pos;
    const int first = pos - n_prev;
    const size_t cache_base = ((size_t)b * a.KV + g) * a.cap;
    const __nv_bfloat16* kcg = a.kc + cache_base * kAD;
    const __nv_bfloat16* vcg = a.vc + cache_base * kAD;
    const int n_tiles = (n_prev + kATile - 1) / kATile;
    auto kbuf = [&](int st) { return asmem + (size_t)st * 2 * kATileBytes; };
    auto vbuf = [&](int st) { return asmem + (size_t)st * 2 * kATileBytes + kATileBytes; };

    // rows past the window's end are zero-filled: their probabilities are 0
    // and 0 * (stale bits) must not make a NaN
    // one modulo per tile: a tile's 64 rows wrap the ring at most once (cap >= 64
    // whenever a window is cached: cap >= window; full attention: cap > pos)
    auto load_tile = [&](int tile, int st) {
        const int p0 = first + tile * kATile;
        const int s0 = p0 % a.cap;
        uint8_t* kd = kbuf(st);
        uint8_t* vd = vbuf(st);
        for (int i = threadIdx.x; i < kATile * 16; i += blockDim.x) {
            const int r = i >> 4, c = i & 15;
            if (p0 + r < pos) {
                int slot = s0 + r;
                while (slot >= a.cap) slot -= a.cap;
                cp_async16(kd + r * kARow + c * 16, kcg + (size_t)slot * kAD + c * 8);
                cp_async16(vd + r * kARow + c * 16, vcg + (size_t)slot * kAD + c * 8);
            } else {
                *reinterpret_cast<uint4*>(kd + r * kARow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(vd + r * kARow + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int t = 0; t < kAStages - 1; ++t)
        if (t < n_tiles) load_tile(t, t); else cp_async_commit();

    // this warp's query head, and (warp 0) the current key and value
    float q[4];
    {
        const __nv_bfloat16* qr = a.q + ((size_t)b * a.H + h) * kAD;
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = __bfloat162float(qr[lane + 32 * i]);
        norm_rope(q, a.wq, lane, pos, a);
#pragma unroll
        for (int i = 0; i < 4; ++i) sh.qs[warp][lane + 32 * i] = q[i];
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
            sh.kcur[lane + 32 * i] = kv[i];
            sh.vcur[lane + 32 * i] = __bfloat162float(vr[lane + 32 * i]);
        }
    }
    __syncthreads();
    // B fragments of Q^T (k = dimension, n = head) for the 8 k-steps: the hi
    // part for warps 0-3, the lo part for warps 4-7
    const int part = warp >> 2, mt = warp & 3;
    uint32_t qb[8][2];
#pragma unroll
    for (int st = 0; st < 8; ++st) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int dim = 16 * st + 2 * cq + 8 * r;
            uint32_t hi, lo;
            split_bf16x2(sh.qs[gq][dim], sh.qs[gq][dim + 1], hi, lo);
            qb[st][r] = part ? lo : hi;
        }
    }
    __syncthreads();   // qs is read; the tile loop reuses its memory for the scores

    const float scale = rsqrtf((float)kAD);   // 1/sqrt(128), exact: 2^-3.5 rounded once
    float m = -INFINITY, l = 0.f;             // warp h's running max and sum (every lane)
    float acc[4] = {0.f, 0.f, 0.f, 0.f};      // O^T: dims 16 w + gq (+8), heads 2 cq (+1)
    const int d0 = 16 * warp;
    for (int tile = 0; tile < n_tiles; ++tile) {
        const int stg = tile % kAStages;
        cp_async_wait<kAStages - 2>();
        __syncthreads();   // the tile has landed; every warp is done with the previous tile
        if (tile + kAStages - 1 < n_tiles) load_tile(tile + kAStages - 1, (tile + kAStages - 1) % kAStages);
        else cp_async_commit();
        const int p0 = first + tile * kATile;
        const int nk = min(kATile, pos - p0);
        const uint8_t* kt = kbuf(stg);
        const uint8_t* vt = vbuf(stg);
        // scores of keys 16 mt .. 16 mt + 15 against the 8 heads (one Q part)
        {
            float sacc[4] = {0.f, 0.f, 0.f, 0.f};
            const int j = lane >> 3, r = lane & 7;
            const uint8_t* rowp = kt + (size_t)(16 * mt + r + 8 * (j & 1)) * kARow + 16 * (j >> 1);
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                uint32_t af[4];
                ldsm_x4(af, rowp + 32 * st);
                mma_bf16_16816(sacc, af[0], af[1], af[2], af[3], qb[st][0], qb[st][1]);
            }
            const int k0 = 16 * mt + gq;
            sh.sc[part][2 * cq][k0] = sacc[0];
            sh.sc[part][2 * cq + 1][k0] = sacc[1];
            sh.sc[part][2 * cq][k0 + 8] = sacc[2];
            sh.sc[part][2 * cq + 1][k0 + 8] = sacc[3];
        }
        __syncthreads();
        // softmax update of head `warp`: lane L takes keys 2L, 2L + 1
        {
            float sv[2];
            const float2 s_hi = *reinterpret_cast<const float2*>(&sh.sc[0][warp][2 * lane]);
            const float2 s_lo = *reinterpret_cast<const float2*>(&sh.sc[1][warp][2 * lane]);
            sv[0] = 2 * lane < nk ? (s_hi.x + s_lo.x) * scale : -INFINITY;
            sv[1] = 2 * lane + 1 < nk ? (s_hi.y + s_lo.y) * scale : -INFINITY;
            const float m_new = fmaxf(m, warp_max(fmaxf(sv[0], sv[1])));
            const float corr = expf(m - m_new);   // 0 on the first tile (m = -inf)
            const float p0v = expf(sv[0] - m_new), p1v = expf(sv[1] - m_new);
            l = l * corr + warp_sum(p0v + p1v);
            m = m_new;
            uint32_t hi, lo;
            split_bf16x2(p0v, p1v, hi, lo);
            sh.ph[warp][lane] = hi;
            sh.pl[warp][lane] = lo;
            if (lane == 0) sh.corr[warp] = corr;
        }
        __syncthreads();
        // O^T[dims d0..d0+15][heads] = corr * O^T + V^T . P^T
        {
            const float c0 = sh.corr[2 * cq], c1 = sh.corr[2 * cq + 1];
            acc[0] *= c0;
            acc[1] *= c1;
            acc[2] *= c0;
            acc[3] *= c1;
            const int j = lane >> 3, r = lane & 7;
#pragma unroll
            for (int st = 0; st < 4; ++st) {
                uint32_t af[4];
                ldsm_x4_t(af, vt + (size_t)(16 * st + r + 8 * (j >> 1)) * kARow + 2 * (d0 + 8 * (j & 1)));
                const int pr = 8 * st + cq;
                mma_bf16_16816(acc, af[0], af[1], af[2], af[3], sh.ph[gq][pr], sh.ph[gq][pr + 4]);
                mma_bf16_16816(acc, af[0], af[1], af[2], af[3], sh.pl[gq][pr], sh.pl[gq][pr + 4]);
            }
        }
    }
    cp_async_wait<0>();
    // the current token (unrounded), then the sink (denominator only), per head
    {
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) dot = fmaf(q[i], sh.kcur[lane + 32 * i], dot);
        const float sc = warp_sum(dot) * scale;
        const float m1 = fmaxf(m, sc);
        const float corr1 = expf(m - m1);
        const float pc = expf(sc - m1);
        const float l1 = l * corr1 + pc;
        const float sk = __ldg(a.sinks + h);
        const float m2 = fmaxf(m1, sk);
        const float corr2 = expf(m1 - m2);
        const float l2 = l1 * corr2 + expf(sk - m2);
        if (lane == 0) {
            sh.fin_a[warp] = corr1 * corr2;
            sh.fin_b[warp] = pc * corr2;
            sh.fin_inv[warp] = 1.0f / l2;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int head = 2 * cq + (i & 1), dim = d0 + gq + 8 * (i >> 1);
        const float o = (acc[i] * sh.fin_a[head] + sh.fin_b[head] * sh.vcur[dim]) * sh.fin_inv[head];
        a.out[((size_t)b * a.H + g * kAGroup + head) * kAD + dim] = __float2bfloat16_rn(o);
    }
    // store the current key and value, bf16, in the position's slot (outside
    // the window that was read: cap >= window)
    if (warp == 0) {
        const size_t slot = (size_t)(pos % a.cap);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a.kc[(cache_base + slot) * kAD + lane + 32 * i] = __float2bfloat16_rn(sh.kcur[lane + 32 * i]);
            a.vc[(cache_base + slot) * kAD + lane + 32 * i] = __float2bfloat16_rn(sh.vcur[lane + 32 * i]);
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
    // frequencies theta^(-i/64) in turns per position, as 64-bit fractions
    // (long double: 64 significant bits on the host)
    for (int i = 0; i < kAD / 2; ++i) {
        const long double f = powl((long double)cfg->rope_theta, -(long double)i / (kAD / 2));
        const long double t = f / (2.0L * 3.14159265358979323846264338327950288L);   // turns per position
        const long double frac = t - floorl(t);
        a.rope_turns[i] = (unsigned long long)(frac * 18446744073709551616.0L);
    }
    a.eps = cfg->eps;
    static bool opted_in = false;   // the attribute is per device function, set once
    if (!opted_in) {
        if (cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kASmem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
                cudaSuccess) {
            cudaGetLastError();
            return FLINT_ECUDA;
        }
        opted_in = true;
    }
    attn_decode_kernel<<<dim3(cfg->n_kv, B), 256, kASmem, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? FLINT_OK : FLINT_ECUDA;
}
