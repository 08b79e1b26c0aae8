// Single-launch decode of one MoE layer for T <= 2 tokens.
//
// Decode streams the selected experts' weights once and does little
// arithmetic on them ("Recursive Flint 40B-A2.5B", section "The architecture
// is an argument about memory bandwidth"), so the step is bound by HBM and by
// the latency of its three dependent phases. One persistent kernel, one CTA
// per SM, runs them with two grid barriers instead of separate launches, and
// every weight slab a CTA needs is requested with 1-D bulk copies (TMA) into
// shared memory as soon as its address is known:
//
//   P0  router logits (each CTA a slice of W_r) -> arrive at the barrier;
//       while it completes, stage x as fp16 and run the shared expert's
//       gate/up (routing-independent, its slab requested at kernel start);
//       the shared expert's down slab is prefetched for P2.
//   --- grid barrier ---
//   P1  every CTA takes the top-6 of the logits itself (no broadcast needed),
//       prefetches the routed experts' down slabs for its P2 rows, then runs
//       its routed gate/up units (16 rows of one expert, full K) from bulk-
//       copied slabs.
//   --- grid barrier ---
//   P2  down projection of 16 output rows for every active expert, weighted
//       combine (shared first, then slots 0..k-1) and bf16 output.
//
// Arithmetic matches the multi-kernel path: weights decoded in registers
// (NVFP4 to exact fp16 products, q4_1 to its exact codes with d and m applied
// per 32-element block to the fp32 accumulator), activations fp16 with a
// power-of-two scale per token (x) or per (token, slot) row (h), mma.sync
// m16n8k16 with fp32 accumulation.
#include "kernels.cuh"
#include "tiles.cuh"
#include "topk.cuh"

namespace flint {

namespace {

constexpr int kFThreads = 512;   // 16 warps
constexpr size_t kMaxSmemOptin = 232448;          // 227 KiB of shared memory per CTA (static + dynamic)
constexpr size_t kFusedDynSmemMax = kMaxSmemOptin - 1024;   // dynamic part; the kernel's static part is < 1 KiB
constexpr int kFWarps = kFThreads / 32;

struct FusedArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* tscale;
    const float* router;
    const float* bias;
    size_t cpm, spm;            // bytes of codes / scales per matrix
    const __nv_bfloat16* x;
    __nv_bfloat16* out;
    const __nv_bfloat16* residual;
    int T, d, f, E, k;
    float* logits;              // [T][E]
    float* h;                   // [T][k+1][f] fp32, slot k = shared expert
    unsigned long long* bar_count;   // grid-barrier arrival counter
    uint32_t* status;
    int n_slots;                // gate/up unit slots in shared memory
    // shared-memory layout (byte offsets)
    int off_slots, unit_bytes, off_down, down_bytes, off_acc, off_x16, off_h16, off_misc, off_xbf, off_ts;
    int ts_bytes;               // bytes of the tensor-scale array copied to shared memory
    // the next layer of a stack (null: none): its routing-independent weights
    // are prefetched into L2 while this layer finishes
    const uint8_t* next_codes;
    const uint8_t* next_scales;
    const float* next_router;
};

struct Pair {
    int t, j;   // token, slot (j == k: shared expert)
};

__device__ __forceinline__ void lds_b16(const __half* p, uint32_t (&b)[16]) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = q[i];
        b[4 * i + 0] = v.x;
        b[4 * i + 1] = v.y;
        b[4 * i + 2] = v.z;
        b[4 * i + 3] = v.w;
    }
}

// Issue the four bulk copies of one gate/up half-unit (8-row group g8 of gate
// and of up of expert e, full K) into slot memory `dst`: gate codes, up codes
// (KT tiles of 512 B each), gate scales, up scales; completing on `bar`.
template <int WFMT>
__device__ void issue_half(const FusedArgs& a, int e, int g8, uint8_t* dst, uint64_t* bar) {
    const int KT = a.d >> 7;
    const int S = WFMT == 0 ? 64 : 128;
    const uint32_t cbytes = (uint32_t)KT * 512u, sbytes = (uint32_t)KT * S;
    mbar_arrive_expect_tx(bar, 2 * (cbytes + sbytes));
    for (int m = 0; m < 2; ++m) {
        bulk_g2s(dst + m * cbytes, a.codes + ((size_t)e * 3 + m) * a.cpm + (size_t)g8 * cbytes, cbytes, bar);
        bulk_g2s(dst + 2 * cbytes + m * sbytes, a.scales + ((size_t)e * 3 + m) * a.spm + (size_t)g8 * sbytes, sbytes,
                 bar);
    }
}

// Issue the two bulk copies of the down slab (16 output rows, full f) of
// expert e for output tile r16.
template <int WFMT>
__device__ void issue_down(const FusedArgs& a, int e, int r16, uint8_t* dst, uint64_t* bar) {
    const int KT = a.f >> 7;
    const int S = WFMT == 0 ? 64 : 128;
    const uint32_t cbytes = 2u * KT * 512u, sbytes = 2u * KT * S;
    bulk_g2s(dst, a.codes + ((size_t)e * 3 + 2) * a.cpm + (size_t)(2 * r16) * KT * 512, cbytes, bar);
    bulk_g2s(dst + cbytes, a.scales + ((size_t)e * 3 + 2) * a.spm + (size_t)(2 * r16) * KT * S, sbytes, bar);
}

constexpr int kMaxWaveUnits = 3;   // gate/up half-units computed together (one wave of slots)

// One gate/up half-unit held in shared memory: slab, expert, 8-row group, and
// its (token, slot) pairs.
struct UnitRef {
    const uint8_t* slab;
    int e, g8;
    const Pair* pairs;
    int np;
};

// Gate/up of up to kMaxWaveUnits half-units. The MMA's 16 A rows are the
// half-unit's 8 gate rows (rows 0-7) and the same 8 up rows (rows 8-15), so
// one m16n8k16 chain yields both projections. Warp w takes k-tiles w, w+16,
// ... of each half-unit in turn and leaves its partial in red[unit][warp];
// then 64 threads per half-unit reduce the 16 warp partials in warp order and
// write h = silu(g) * u (fp32) for its 8 rows. The unit loop is not unrolled:
// this code runs once per launch, so its size (instruction fetch), not its
// instruction-level parallelism, is what costs.
template <int WFMT>
__device__ void gateup_units(const FusedArgs& a, const UnitRef* units, int n_units, const __half* x16s,
                             const float* xinv, const float* tss, float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KT = a.d >> 7;
    const int S = WFMT == 0 ? 64 : 128;
#pragma unroll 1
    for (int v = 0; v < n_units; ++v) {
        const UnitRef un = units[v];
        const uint8_t* cg = un.slab;
        const uint8_t* cu = un.slab + KT * 512;
        const uint8_t* sg = un.slab + 2 * KT * 512;
        const uint8_t* su = sg + KT * S;
        const int tb = (g < un.np) ? un.pairs[g].t : -1;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int kt = warp; kt < KT; kt += kFWarps) {
            const uint4 wg = *reinterpret_cast<const uint4*>(cg + kt * 512 + lane * 16);
            const uint4 wu = *reinterpret_cast<const uint4*>(cu + kt * 512 + lane * 16);
            const TileScales<WFMT> sc = lds_scales<WFMT>(sg + kt * S, su + kt * S, g);
            uint32_t b[16];
            if (tb >= 0) {
                lds_b16(x16s + (size_t)tb * a.d + kt * 128 + c * 32, b);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) b[i] = 0u;
            }
            uint32_t fa[8][4];
            decode_tile<WFMT>(wg, wu, sc, fa);
            float sx[4][2];
            if constexpr (WFMT == 1) block_sums_q41(b, sx);
            mma_k128<WFMT>(acc, fa, b, sc, sx);
        }
        *reinterpret_cast<float4*>(red + (size_t)(v * kFWarps + warp) * 128 + lane * 4) =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
    __syncthreads();
    if (threadIdx.x < 64 * n_units) {
        // thread i of unit v: fragment lane ln = i/2, column 2*(ln%4) + i%2,
        // row ln/4; its gate sum is element ln*4 + (i%2), its up sum element + 2
        const int v = threadIdx.x >> 6, i = threadIdx.x & 63;
        const UnitRef& un = units[v];
        const int ln = i >> 1, jj = i & 1;
        const int n = 2 * (ln & 3) + jj;
        if (n < un.np) {
            const float* rv = red + (size_t)v * kFWarps * 128 + ln * 4 + jj;
            float sg_ = 0.f, su_ = 0.f;
#pragma unroll
            for (int w = 0; w < kFWarps; ++w) {
                sg_ += rv[w * 128];
                su_ += rv[w * 128 + 2];
            }
            const Pair p = un.pairs[n];
            const float gv = sg_ * tss[un.e * 3 + 0] * xinv[p.t];
            const float uv = su_ * tss[un.e * 3 + 1] * xinv[p.t];
            const float hv = gv / (1.0f + expf(-gv)) * uv;
            const int row = un.g8 * 8 + (ln >> 2);
            a.h[((size_t)p.t * (a.k + 1) + p.j) * a.f + row] = hv;
        }
    }
    __syncthreads();
}

template <int WFMT, int TT>
__global__ void __launch_bounds__(kFThreads, 1) decode_fused_kernel(FusedArgs a) {
    // TT: the token count, a template parameter so that the per-token loops
    // compile to straight code for exactly that count
    static_assert(TT >= 1 && TT <= kFusedMaxT, "token count");
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int G = gridDim.x, b = blockIdx.x;
    constexpr int T = TT;
    const int d = a.d, f = a.f, E = a.E, k = a.k;
    const int KTf = f >> 7;
    const int units_per_expert = f >> 3;                 // 8-row half-units
    const int down_tiles = d >> 4;
    const int down_tile = b - (G - down_tiles);          // the last d/16 CTAs own output tiles
    const int shared_unit = G - 1 - b;                   // the last f/8 CTAs do the shared gate/up

    uint8_t* slots = smem + a.off_slots;
    uint8_t* down = smem + a.off_down;
    float* acc = reinterpret_cast<float*>(smem + a.off_acc);
    __half* x16s = reinterpret_cast<__half*>(smem + a.off_x16);
    __half* h16s = reinterpret_cast<__half*>(smem + a.off_h16);
    uint8_t* misc = smem + a.off_misc;
    const __nv_bfloat16* xbf = reinterpret_cast<const __nv_bfloat16*>(smem + a.off_xbf);
    const float* tss = reinterpret_cast<const float*>(smem + a.off_ts);
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);              // [n_slots + 4]
    uint64_t* bar_router = bars + a.n_slots;
    uint64_t* bar_dshared = bars + a.n_slots + 1;
    uint64_t* bar_drouted = bars + a.n_slots + 2;
    uint64_t* bar_x = bars + a.n_slots + 3;
    float* xinv = reinterpret_cast<float*>(misc + 128);              // [2]
    float* hinv = xinv + 4;                                          // [2*(k+1)] <= 18
    float* rpart = hinv + 20;                                        // [16][2]
    float* lg = rpart + 32;                                          // [2][256]
    int* sel = reinterpret_cast<int*>(lg + 2 * 256);                 // [2][8]
    float* wsel = reinterpret_cast<float*>(sel + 16);                // [2][8]
    int* act = reinterpret_cast<int*>(wsel + 16);                    // [17] active experts (routed)
    int* act_np = act + 17;                                          // [17]
    Pair* act_pairs = reinterpret_cast<Pair*>(act_np + 17);          // [17][2]
    int* nact = reinterpret_cast<int*>(act_pairs + 34);              // [1]
    Pair* shared_pairs = reinterpret_cast<Pair*>(nact + 2);          // [2]
    float* bias_s = reinterpret_cast<float*>(shared_pairs + 2);      // [2]
    int* cmap = reinterpret_cast<int*>(bias_s + 2);                  // [2][8]

    bool ok = true;
    uint32_t slot_phase = 0;   // bit s: parity of slot s's next completion
    // thread 0 (the only thread that issues bulk copies): bit i of pend = a
    // copy was issued on barrier bars[i], whose phase of parity bit i of
    // pend_par it completes. No copy is issued once a wait has given up, so
    // at exit drain() waits (bounded) for exactly the copies that may still
    // be in flight and none of them writes shared memory after the CTA is gone.
    uint32_t pend = 0, pend_par = 0;
    auto mark_issued = [&](int i, uint32_t parity) {
        pend |= 1u << i;
        pend_par = (pend_par & ~(1u << i)) | (parity << i);
    };
    auto drain = [&]() {
        if (threadIdx.x == 0) {
#pragma unroll 1
            for (int i = 0; i < a.n_slots + 4; ++i)
                if ((pend >> i) & 1u) mbar_wait_bounded(bars + i, (pend_par >> i) & 1u, a.status);
        }
    };
    // CTA-uniform bounded wait: every thread waits, and the CTA proceeds only
    // if all of them saw the phase complete.
    auto wait_all = [&](uint64_t* bar, uint32_t ph) {
        const bool w = ok ? mbar_wait_bounded(bar, ph, a.status) : false;
        ok = __syncthreads_and(w ? 1 : 0) != 0;
    };

    if (threadIdx.x == 0) {
#pragma unroll 1
        for (int i = 0; i < a.n_slots + 4; ++i) mbar_init(bars + i, 1);
        mbar_fence_init();
    }
    __syncthreads();

    // ------------------------------------------------------------------ P0
    // router slice: experts b, b+G, ... (at most 2 rows held in slot 0); the
    // shared expert's gate/up unit (slot n_slots-1) and down slab are
    // prefetched now and used in P1 / P2.
    int n_re = 0;
    for (int e = b; e < E; e += G) ++n_re;
    const int shared_slot = a.n_slots - 1;
    const bool has_shared = shared_unit >= 0 && shared_unit < units_per_expert;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar_x, (uint32_t)(T * d * 2 + a.ts_bytes));
        bulk_g2s(smem + a.off_xbf, a.x, (uint32_t)(T * d * 2), bar_x);
        bulk_g2s(smem + a.off_ts, a.tscale, (uint32_t)a.ts_bytes, bar_x);
        mark_issued(a.n_slots + 3, 0u);
        if (n_re > 0) {
            mbar_arrive_expect_tx(bar_router, (uint32_t)(n_re * d * 4));
#pragma unroll 1
            for (int i = 0; i < n_re; ++i)
                bulk_g2s(slots + (size_t)i * d * 4, a.router + (size_t)(b + i * G) * d, d * 4, bar_router);
            mark_issued(a.n_slots, 0u);
        }
        if (has_shared) {
            issue_half<WFMT>(a, E, shared_unit, slots + (size_t)shared_slot * a.unit_bytes, bars + shared_slot);
            mark_issued(shared_slot, 0u);
        }
        if (down_tile >= 0) {
            mbar_arrive_expect_tx(bar_dshared, (uint32_t)a.down_bytes);
            issue_down<WFMT>(a, E, down_tile, down, bar_dshared);
            mark_issued(a.n_slots + 1, 0u);
        }
    }
    if (threadIdx.x >= 32 && threadIdx.x < 32 + n_re) bias_s[threadIdx.x - 32] = __ldg(a.bias + b + (threadIdx.x - 32) * G);
    GridSync gsync = grid_sync_init(a.bar_count, (uint32_t)G);   // includes a __syncthreads
    wait_all(bar_x, 0);
    if (threadIdx.x < T) {
        shared_pairs[threadIdx.x].t = threadIdx.x;
        shared_pairs[threadIdx.x].j = k;
    }
    // router logits of this CTA's experts
    if (n_re > 0) {
        wait_all(bar_router, 0);
        const int i = warp / 8, part = warp % 8;    // 8 warps per expert row
        const int seg = d / 8;                      // elements per warp (multiple of 16)
        float accv[2] = {0.f, 0.f};
        if (ok && i < n_re) {
            const float* wr = reinterpret_cast<const float*>(slots) + (size_t)i * d + part * seg;
#pragma unroll 1
            for (int q = lane * 4; q < seg; q += 128) {
                const float4 wv = *reinterpret_cast<const float4*>(wr + q);
                for (int t = 0; t < T; ++t) {
                    const __nv_bfloat16* xr = xbf + (size_t)t * d + part * seg + q;
                    const uint2 raw = *reinterpret_cast<const uint2*>(xr);
                    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
                    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
                    float s = accv[t];
                    s = fmaf(wv.x, __low2float(p0), s);
                    s = fmaf(wv.y, __high2float(p0), s);
                    s = fmaf(wv.z, __low2float(p1), s);
                    s = fmaf(wv.w, __high2float(p1), s);
                    accv[t] = s;
                }
            }
        }
        for (int t = 0; t < T; ++t) {
            const float s = warp_sum(accv[t]);
            if (lane == 0) rpart[warp * 2 + t] = s;
        }
        __syncthreads();
        if (threadIdx.x < n_re * T) {
            const int ii = threadIdx.x / T, t = threadIdx.x % T;
            float s = 0.f;
            for (int p = 0; p < 8; ++p) s += rpart[(ii * 8 + p) * 2 + t];
            const int e = b + ii * G;
            a.logits[(size_t)t * E + e] = s + bias_s[ii];
        }
    }
    grid_arrive(gsync);
    // while the barrier completes: stage the hidden states as fp16, scaled
    // per token, fragment-permuted
    // (thread i holds elements 4(i + 512q) .. +3, stored as half2 pairs)
    for (int t = 0; t < T; ++t) {
        float xv[2][4];
        float amax = 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = (threadIdx.x + q * kFThreads) * 4;
            uint2 raw = make_uint2(0u, 0u);
            if (i < d) raw = *reinterpret_cast<const uint2*>(xbf + (size_t)t * d + i);
            const float2 p0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
            const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
            xv[q][0] = p0.x;
            xv[q][1] = p0.y;
            xv[q][2] = p1.x;
            xv[q][3] = p1.y;
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(p0.x), fabsf(p0.y)), fmaxf(fabsf(p1.x), fabsf(p1.y))));
        }
        amax = warp_max(amax);
        if (lane == 0) rpart[warp] = amax;
        __syncthreads();
        float m = 0.f;
#pragma unroll
        for (int w = 0; w < kFWarps; ++w) m = fmaxf(m, rpart[w]);
        const float mult = f16_range_mult(m);
        __half2* xrow = reinterpret_cast<__half2*>(x16s + (size_t)t * d);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = (threadIdx.x + q * kFThreads) * 4;
            if (i < d) {
                __half2* tile = xrow + ((i & ~127) >> 1);
                tile[kperm_pos(i & 127) >> 1] = __floats2half2_rn(xv[q][0] * mult, xv[q][1] * mult);
                tile[kperm_pos((i & 127) + 2) >> 1] = __floats2half2_rn(xv[q][2] * mult, xv[q][3] * mult);
            }
        }
        if (threadIdx.x == 0) xinv[t] = 1.0f / mult;
        __syncthreads();
    }
    if (!grid_wait(gsync, a.status)) ok = false;

    // ------------------------------------------------------------------ P1
    // top-k of every token, computed by every CTA from the logits in L2
#pragma unroll 1
    for (int i = threadIdx.x; i < T * E; i += kFThreads) lg[i] = __ldcg(a.logits + i);
    __syncthreads();
    if (warp < T) topk_warp<false>(lg + warp * E, E, k, sel + warp * 8, wsel + warp * 8, b == 0 ? a.status : nullptr);
    __syncthreads();
    if (T == 1) {
        // one token: its k experts are distinct, one pair each
        if (threadIdx.x < k) {
            const int j = threadIdx.x;
            act[j] = sel[j];
            act_np[j] = 1;
            act_pairs[j * 2] = Pair{0, j};
            cmap[j] = (j + 1) * 4;
            if (j == 0) *nact = k;
        }
    } else if (warp == 0) {
        // distinct routed experts and their (token, slot) pairs, by one warp:
        // entry i = t*k + j; an entry is the first of its expert if no earlier
        // entry has the same expert; experts are numbered in first-occurrence
        // order (the order does not change any result).
        const int n = T * k;
        const int t = lane / k, j = lane - (lane / k) * k;
        const int e = lane < n ? sel[t * 8 + j] : -1 - lane;
        int first = lane, p = 0;
        for (int i = 0; i < n; ++i) {
            const int ei = __shfl_sync(0xffffffffu, e, i);
            if (i < lane && ei == e) {
                if (first == lane) first = i;
                ++p;
            }
        }
        const uint32_t firsts = __ballot_sync(0xffffffffu, lane < n && first == lane);
        const int q = __popc(firsts & ((1u << first) - 1u));   // dense index of this entry's expert
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (lane < n) {
            if (first == lane) {
                act[q] = e;
                act_np[q] = __popc(same);
            }
            act_pairs[q * 2 + p] = Pair{t, j};
            cmap[t * 8 + j] = (q + 1) * 4 + p;
        }
        if (lane == 0) *nact = __popc(firsts);
    }
    __syncthreads();
    const int na = *nact;
    const int n_units = na * units_per_expert;
    // routed gate/up units u = b, b+G, ..., in waves of n_slots-1 slots; the
    // shared expert's unit (its slab landed in P0) is computed while the
    // first wave's slabs are in flight
    const int n_rs = a.n_slots - 1;
    // one gateup_units call site: each pass computes either the shared
    // half-unit or one wave of routed half-units
    bool shared_pending = has_shared, wave_issued = false;
    for (int u0 = b;;) {
        if (!wave_issued && u0 < n_units && ok) {
            __syncthreads();   // the previous wave's slots have been read
            if (threadIdx.x == 0) {
                fence_proxy_async_smem();
#pragma unroll 1
                for (int s2 = 0; s2 < n_rs; ++s2) {
                    const int u = u0 + s2 * G;
                    if (u < n_units) {
                        issue_half<WFMT>(a, act[u / units_per_expert], u % units_per_expert,
                                         slots + (size_t)s2 * a.unit_bytes, bars + s2);
                        mark_issued(s2, (slot_phase >> s2) & 1u);
                    }
                }
            }
            wave_issued = true;
        }
        UnitRef wave[kMaxWaveUnits];
        int nw = 0;
        if (shared_pending) {
            wait_all(bars + shared_slot, 0);
            wave[nw++] = UnitRef{slots + (size_t)shared_slot * a.unit_bytes, E, shared_unit, shared_pairs, T};
            shared_pending = false;
        } else if (u0 < n_units) {
#pragma unroll 1
            for (int s2 = 0; s2 < n_rs; ++s2) {
                const int u = u0 + s2 * G;
                if (u >= n_units) break;
                const uint32_t ph = (slot_phase >> s2) & 1u;
                wait_all(bars + s2, ph);
                slot_phase ^= 1u << s2;
                const int q = u / units_per_expert;
                wave[nw++] = UnitRef{slots + (size_t)s2 * a.unit_bytes, act[q], u % units_per_expert,
                                     act_pairs + q * 2, act_np[q]};
            }
            u0 += G * n_rs;
            wave_issued = false;
        } else {
            break;
        }
        if (ok && nw > 0) gateup_units<WFMT>(a, wave, nw, x16s, xinv, tss, acc);
    }
    // routed down slabs for this CTA's output tile (slab 0 is the shared
    // expert), requested once the gate/up slabs have landed so that they do
    // not compete with them; they are needed only after the next barrier
    if (threadIdx.x == 0 && down_tile >= 0 && na > 0 && ok) {
        mbar_arrive_expect_tx(bar_drouted, (uint32_t)(na * a.down_bytes));
#pragma unroll 1
        for (int q = 0; q < na; ++q)
            issue_down<WFMT>(a, act[q], down_tile, down + (size_t)(1 + q) * a.down_bytes, bar_drouted);
        mark_issued(a.n_slots + 2, 0u);
    }
    if (!grid_sync(gsync, a.status)) ok = false;

    // ------------------------------------------------------------------ P2
    // the next layer's P0 reads (its router rows, shared half-unit and shared
    // down slab of this CTA) do not depend on this layer's output: request
    // them into L2 now so that they are not DRAM round trips there
    if (threadIdx.x == 0 && a.next_router != nullptr) {
#pragma unroll 1
        for (int i = 0; i < n_re; ++i) bulk_prefetch_l2(a.next_router + (size_t)(b + i * G) * d, d * 4);
        const int KT = d >> 7;
        const int S = WFMT == 0 ? 64 : 128;
        if (has_shared) {
            for (int m = 0; m < 2; ++m) {
                bulk_prefetch_l2(a.next_codes + ((size_t)E * 3 + m) * a.cpm + (size_t)shared_unit * KT * 512, KT * 512);
                bulk_prefetch_l2(a.next_scales + ((size_t)E * 3 + m) * a.spm + (size_t)shared_unit * KT * S, KT * S);
            }
        }
        if (down_tile >= 0) {
            bulk_prefetch_l2(a.next_codes + ((size_t)E * 3 + 2) * a.cpm + (size_t)(2 * down_tile) * KTf * 512,
                             2 * KTf * 512);
            bulk_prefetch_l2(a.next_scales + ((size_t)E * 3 + 2) * a.spm + (size_t)(2 * down_tile) * KTf * S,
                             2 * KTf * S);
        }
    }
    if (down_tile < 0) {
        drain();
        return;
    }
    // stage h rows as fp16 with a power-of-two scale per (token, slot) row
    const int n_rows = T * (k + 1);
    // (lane l holds elements 4(32q + l) .. +3; pairs stay adjacent under the
    // fragment permutation, so they are stored as half2)
    const int nq = f >> 7;
    for (int r = warp; r < n_rows; r += kFWarps) {
        const float4* hr = reinterpret_cast<const float4*>(a.h + (size_t)r * f);
        float4 hv[8];
        float amax = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            hv[q] = q < nq ? __ldcg(hr + q * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(hv[q].x), fabsf(hv[q].y)), fmaxf(fabsf(hv[q].z), fabsf(hv[q].w))));
        }
        amax = warp_max(amax);
        const float mult = f16_range_mult(amax);
        __half2* hrow = reinterpret_cast<__half2*>(h16s + (size_t)r * f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (q < nq) {
                const int i = (q * 32 + lane) * 4;
                __half2* tile = hrow + ((i & ~127) >> 1);
                tile[kperm_pos(i & 127) >> 1] = __floats2half2_rn(hv[q].x * mult, hv[q].y * mult);
                tile[kperm_pos((i & 127) + 2) >> 1] = __floats2half2_rn(hv[q].z * mult, hv[q].w * mult);
            }
        }
        if (lane == 0) hinv[r] = 1.0f / mult;
    }
    wait_all(bar_dshared, 0);
    if (na > 0) wait_all(bar_drouted, 0);
    drain();   // returns at once unless a wait above gave up
    // down products: warps 2q and 2q+1 (slab q = shared, then routed) run the
    // two halves of the k-tiles -> acc[q][half][16 rows][8 pairs]
    const int S = WFMT == 0 ? 64 : 128;
    const int kt_half = (KTf + 1) / 2;
#pragma unroll 1
    for (int it = warp; it < 2 * (na + 1) && ok; it += kFWarps) {
        const int q = it >> 1, hf = it & 1;
        const uint8_t* slab = down + (size_t)q * a.down_bytes;
        const uint8_t* cd = slab;
        const uint8_t* sd = slab + 2 * KTf * 512;
        const int np = q == 0 ? T : act_np[q - 1];
        const Pair* pp = q == 0 ? shared_pairs : act_pairs + (q - 1) * 2;
        const int hrow = g < np ? pp[g].t * (k + 1) + pp[g].j : -1;
        float cacc[4] = {0.f, 0.f, 0.f, 0.f};
        const int kt1 = min(KTf, (hf + 1) * kt_half);
#pragma unroll 1
        for (int kt = hf * kt_half; kt < kt1; ++kt) {
            const uint4 wg = *reinterpret_cast<const uint4*>(cd + kt * 512 + lane * 16);
            const uint4 wh = *reinterpret_cast<const uint4*>(cd + (KTf + kt) * 512 + lane * 16);
            const TileScales<WFMT> sc = lds_scales<WFMT>(sd + kt * S, sd + (KTf + kt) * S, g);
            uint32_t bfr[16];
            if (hrow >= 0) {
                lds_b16(h16s + (size_t)hrow * f + kt * 128 + c * 32, bfr);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) bfr[i] = 0u;
            }
            uint32_t fa[8][4];
            decode_tile<WFMT>(wg, wh, sc, fa);
            float sx[4][2];
            if constexpr (WFMT == 1) block_sums_q41(bfr, sx);
            mma_k128<WFMT>(cacc, fa, bfr, sc, sx);
        }
        float* dst = acc + (size_t)it * 128;
        dst[g * 8 + 2 * c] = cacc[0];
        dst[g * 8 + 2 * c + 1] = cacc[1];
        dst[(g + 8) * 8 + 2 * c] = cacc[2];
        dst[(g + 8) * 8 + 2 * c + 1] = cacc[3];
    }
    __syncthreads();
    // combine: out[t][row] = bf16( y_shared + sum_j w_j y_j ), fixed order
    if (threadIdx.x < T * 16 && ok) {
        const int t = threadIdx.x / 16, rr = threadIdx.x % 16;
        const int orow = down_tile * 16 + rr;
        float v = (acc[rr * 8 + t] + acc[128 + rr * 8 + t]) * tss[E * 3 + 2] * hinv[t * (k + 1) + k];
        for (int j = 0; j < k; ++j) {
            const int e = sel[t * 8 + j];
            const int qp = cmap[t * 8 + j];
            const float* aq = acc + (size_t)(qp >> 2) * 256 + rr * 8 + (qp & 3);
            const float y = aq[0] + aq[128];
            v += wsel[t * 8 + j] * (y * tss[e * 3 + 2] * hinv[t * (k + 1) + j]);
        }
        __nv_bfloat16 o = __float2bfloat16_rn(v);
        if (a.residual != nullptr) {
            const float r = __bfloat162float(a.residual[(size_t)t * d + orow]);
            o = __float2bfloat16_rn(r + __bfloat162float(o));
        }
        a.out[(size_t)t * d + orow] = o;
    }
}


// ---------------------------------------------------------------------------
// The decode stack in one launch: all layers of flint_moe_forward_stack for
// T <= 2 tokens, x <- bf16(x + MoE_l(x)) for l = 0 .. n-1, in one persistent
// cooperative kernel (the one-dispatch decode of the whole forward that the
// Flint blog's Metal megakernel does, section "The quantization recipe is the
// most transferable part"). Per layer two grid barriers instead of a launch:
//
//   P1  every CTA: logits of this layer from the fixed-point accumulators,
//       top-k, routed gate/up half-units (slabs bulk-copied as soon as the
//       experts are known), h to global; requests this CTA's routed down
//       slabs and, for the next layer, its shared half-unit and router slab.
//   --- grid barrier ---
//   P2  the d/16 row-owner CTAs: down products and combine of their 16 rows,
//       x_{l+1} = bf16(x_l + out) in place, then the next layer's router
//       logits restricted to those 16 rows (W_r^T rows, prefetched during P1),
//       added into fixed-point accumulators.
//   --- grid barrier ---
//
// The router logits of layer l+1 are thus sums over the 128 row-owner CTAs of
// partial dot products; they are accumulated as 64-bit integers in units of
// 2^-32 (each partial rounded once to that grid), so the sum is the same
// whatever order the CTAs arrive in and every run gives the same bits. The
// accumulators and their non-finite flags are zero between launches.
// ---------------------------------------------------------------------------
// 2^32 units per logit: a power of two, so the scaling to and from the
// fixed-point grid is exact in fp32 and each conversion rounds once
constexpr float kRaccScale = 4294967296.0f;

struct StackArgs {
    FusedArgs f;                     // shape, shared-memory plan, h scratch, status
    unsigned long long* gbar8;       // grid-barrier counters (GridSync8)
    const StackLayer* layers;        // [n] device table, in stack order
    int n;
    __nv_bfloat16* x;                // [T][d] hidden, updated in place
    unsigned long long* racc;        // [2][kRaccCopies][T][E] fixed-point router logits
    uint32_t* rnf;                   // [2][kRaccCopies][T][E] non-finite partial seen
    int off_rslab;                   // shared-memory offset of the router slab [16][E] fp32
};

// Row owners: partial logits of 16 rows of x (xr[t][r], fp32 of bf16) with the
// router slab (rslab[r][e] = W_r[e][16 dt + r]) into copy `copy` of
// racc/rnf (the owners spread over kRaccCopies copies, so that fewer atomics
// queue on one address; the readers add the copies, exactly).
template <int TT>
__device__ void router_partials(const StackArgs& sa, const float* rslab, const float* xr, int buf, int copy) {
    const int E = sa.f.E;
    for (int i = threadIdx.x; i < TT * E; i += kFThreads) {
        const int t = i / E, e = i - (i / E) * E;
        float p = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) p = fmaf(rslab[r * E + e], xr[t * 16 + r], p);
        const size_t o = (((size_t)buf * kRaccCopies + copy) * TT + t) * E + e;
        if (!(fabsf(p) <= 1.0e9f)) {   // non-finite, or beyond the fixed-point range
            atomicOr(sa.rnf + o, 1u);
        } else {
            const long long q = __float2ll_rn(p * kRaccScale);
            atomicAdd(sa.racc + o, (unsigned long long)q);
        }
    }
}

template <int WFMT, int TT>
__global__ void __launch_bounds__(kFThreads, 1) decode_stack_kernel(StackArgs sa) {
    static_assert(TT >= 1 && TT <= kFusedMaxT, "token count");
    extern __shared__ __align__(128) uint8_t smem[];
    const FusedArgs a0 = sa.f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int G = gridDim.x, b = blockIdx.x;
    constexpr int T = TT;
    const int d = a0.d, f = a0.f, E = a0.E, k = a0.k;
    const int KTf = f >> 7;
    const int units_per_expert = f >> 3;
    const int down_tiles = d >> 4;
    const int down_tile = b - (G - down_tiles);          // the last d/16 CTAs own 16 rows each
    const int shared_unit = G - 1 - b;                   // the last f/8 CTAs do the shared gate/up

    uint8_t* slots = smem + a0.off_slots;
    uint8_t* down = smem + a0.off_down;
    float* acc = reinterpret_cast<float*>(smem + a0.off_acc);
    __half* x16s = reinterpret_cast<__half*>(smem + a0.off_x16);
    __half* h16s = reinterpret_cast<__half*>(smem + a0.off_h16);
    uint8_t* misc = smem + a0.off_misc;
    float* tss = reinterpret_cast<float*>(smem + a0.off_ts);
    float* rslab = reinterpret_cast<float*>(smem + sa.off_rslab);
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);              // [n_slots + 4]
    const int i_rslab = a0.n_slots, i_dshared = a0.n_slots + 1, i_drouted = a0.n_slots + 2;
    float* xinv = reinterpret_cast<float*>(misc + 128);              // [2]
    float* hinv = xinv + 4;                                          // [2*(k+1)] <= 18
    float* rpart = hinv + 20;                                        // [16][2]
    float* lg = rpart + 32;                                          // [2][256]
    int* sel = reinterpret_cast<int*>(lg + 2 * 256);                 // [2][8]
    float* wsel = reinterpret_cast<float*>(sel + 16);                // [2][8]
    int* act = reinterpret_cast<int*>(wsel + 16);                    // [17]
    int* act_np = act + 17;                                          // [17]
    Pair* act_pairs = reinterpret_cast<Pair*>(act_np + 17);          // [17][2]
    int* nact = reinterpret_cast<int*>(act_pairs + 34);              // [1]
    Pair* shared_pairs = reinterpret_cast<Pair*>(nact + 2);          // [2]
    int* cmap = reinterpret_cast<int*>(shared_pairs + 2 + 2);        // [2][8]
    float* xr = reinterpret_cast<float*>(misc + 3072);               // [2][16] x_{l+1} rows of this CTA

    bool ok = true;
    uint32_t ph = 0;   // bit i: parity of the next completion of bars[i] (uniform over the CTA)
    auto wait_bar = [&](int i) {
        const bool w = ok ? mbar_wait_bounded(bars + i, (ph >> i) & 1u, a0.status) : false;
        ph ^= 1u << i;
        ok = __syncthreads_and(w ? 1 : 0) != 0;
    };
    // thread 0 issues every bulk copy; pend/pend_par track the ones that may
    // still be in flight (see decode_fused_kernel)
    uint32_t pend = 0, pend_par = 0;
    auto mark_issued = [&](int i) {
        pend |= 1u << i;
        pend_par = (pend_par & ~(1u << i)) | (((ph >> i) & 1u) << i);
    };
    auto drain = [&]() {
        if (threadIdx.x == 0) {
#pragma unroll 1
            for (int i = 0; i < a0.n_slots + 4; ++i)
                if ((pend >> i) & 1u) mbar_wait_bounded(bars + i, (pend_par >> i) & 1u, a0.status);
        }
    };
    auto args_of = [&](const StackLayer& L) {
        FusedArgs al = a0;
        al.codes = L.codes;
        al.scales = L.scales;
        al.tscale = L.tscale;
        al.bias = L.bias;
        return al;
    };
    // the pointer table entries of the current and the next layer, each
    // loaded one layer ahead so that no request waits on a table read
    StackLayer Lc = sa.layers[0];
    StackLayer Ln = sa.n > 1 ? sa.layers[1] : Lc;

    if (threadIdx.x == 0) {
#pragma unroll 1
        for (int i = 0; i < a0.n_slots + 4; ++i) mbar_init(bars + i, 1);
        mbar_fence_init();
    }
    if (threadIdx.x < T) {
        shared_pairs[threadIdx.x].t = threadIdx.x;
        shared_pairs[threadIdx.x].j = k;
    }
    __syncthreads();
    const int shared_slot = a0.n_slots - 1;
    const bool has_shared = shared_unit >= 0 && shared_unit < units_per_expert;
    const uint32_t rslab_bytes = (uint32_t)(16 * E * 4);

    // ---- prologue: layer 0's routing-independent slabs, and its router
    // logits from the input rows (row owners)
    {
        const FusedArgs al = args_of(Lc);
        if (threadIdx.x == 0) {
            if (has_shared) {
                issue_half<WFMT>(al, E, shared_unit, slots + (size_t)shared_slot * al.unit_bytes, bars + shared_slot);
                mark_issued(shared_slot);
            }
            if (down_tile >= 0) {
                mbar_arrive_expect_tx(bars + i_dshared, (uint32_t)al.down_bytes);
                issue_down<WFMT>(al, E, down_tile, down, bars + i_dshared);
                mark_issued(i_dshared);
                mbar_arrive_expect_tx(bars + i_rslab, rslab_bytes);
                bulk_g2s(rslab, Lc.router_t + (size_t)16 * down_tile * E, rslab_bytes, bars + i_rslab);
                mark_issued(i_rslab);
            }
        }
    }
    GridSync gsync = grid_sync_init(a0.bar_count, (uint32_t)G);   // includes a __syncthreads
    if (down_tile >= 0) {
        if (threadIdx.x < T * 16) {
            const int t = threadIdx.x / 16, r = threadIdx.x % 16;
            xr[t * 16 + r] = __bfloat162float(sa.x[(size_t)t * d + 16 * down_tile + r]);
        }
        wait_bar(i_rslab);
        if (ok) router_partials<T>(sa, rslab, xr, 0, down_tile % kRaccCopies);
    }
    if (!grid_sync(gsync, a0.status)) ok = false;

#pragma unroll 1
    for (int li = 0; li < sa.n && ok; ++li) {
        const FusedArgs al = args_of(Lc);
        const int buf = li & 1;
        const bool last = li + 1 == sa.n;
        const StackLayer Lnn = li + 2 < sa.n ? sa.layers[li + 2] : Ln;   // used from the next layer on
        // ------------------------------------------------------------ P1
        // every independent load of the layer start is issued first: tensor
        // scales, this thread's logit accumulators (all copies) and bias, and
        // its elements of x_l (T <= 2, so at most T*E = 512 logits: one per thread)
        const int n_ts = 3 * (E + 1);
        const float ts0 = threadIdx.x < n_ts ? __ldg(al.tscale + threadIdx.x) : 0.f;
        const float ts1 = threadIdx.x + kFThreads < n_ts ? __ldg(al.tscale + threadIdx.x + kFThreads) : 0.f;
        long long qsum = 0;
        uint32_t nf = 0;
        float bias_v = 0.f;
        if (threadIdx.x < T * E) {
            unsigned long long qv[kRaccCopies];
            uint32_t fv[kRaccCopies];
#pragma unroll
            for (int cpy = 0; cpy < kRaccCopies; ++cpy) {
                const size_t o = (((size_t)buf * kRaccCopies + cpy) * T) * E + threadIdx.x;
                qv[cpy] = __ldcg(sa.racc + o);
                fv[cpy] = __ldcg(sa.rnf + o);
            }
            bias_v = __ldg(al.bias + (threadIdx.x % E));
#pragma unroll
            for (int cpy = 0; cpy < kRaccCopies; ++cpy) {
                qsum += (long long)qv[cpy];
                nf |= fv[cpy];
            }
        }
        uint2 xraw[T][2];
#pragma unroll
        for (int t = 0; t < T; ++t)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i = (threadIdx.x + q * kFThreads) * 4;
                xraw[t][q] = i < d ? __ldcg(reinterpret_cast<const uint2*>(sa.x + (size_t)t * d + i)) : make_uint2(0u, 0u);
            }
        if (threadIdx.x < n_ts) tss[threadIdx.x] = ts0;
        if (threadIdx.x + kFThreads < n_ts) tss[threadIdx.x + kFThreads] = ts1;
        if (threadIdx.x < T * E) {
            const float v = __ll2float_rn(qsum) * (1.0f / kRaccScale) + bias_v;
            lg[(threadIdx.x / E) * 256 + (threadIdx.x % E)] = nf ? __int_as_float(0x7fc00000) : v;
        }
        // the other accumulator is filled by this layer's P2; its last readers
        // finished before the previous layer's barriers
        if (b == 0) {
            for (int i = threadIdx.x; i < kRaccCopies * T * E; i += kFThreads) {
                sa.racc[(size_t)(buf ^ 1) * kRaccCopies * T * E + i] = 0ull;
                sa.rnf[(size_t)(buf ^ 1) * kRaccCopies * T * E + i] = 0u;
            }
        }
        // x_l as fp16, scaled per token, fragment-permuted: staged after the
        // routed slabs have been requested, so that it overlaps their latency
        auto stage_x = [&]() {
            for (int t = 0; t < T; ++t) {
                float xv[2][4];
                float amax = 0.f;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint2 raw = xraw[t][q];
                    const float2 p0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
                    const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
                    xv[q][0] = p0.x;
                    xv[q][1] = p0.y;
                    xv[q][2] = p1.x;
                    xv[q][3] = p1.y;
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(p0.x), fabsf(p0.y)), fmaxf(fabsf(p1.x), fabsf(p1.y))));
                }
                amax = warp_max(amax);
                if (lane == 0) rpart[warp] = amax;
                __syncthreads();
                float m = 0.f;
#pragma unroll
                for (int w = 0; w < kFWarps; ++w) m = fmaxf(m, rpart[w]);
                const float mult = f16_range_mult(m);
                __half2* xrow = reinterpret_cast<__half2*>(x16s + (size_t)t * d);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int i = (threadIdx.x + q * kFThreads) * 4;
                    if (i < d) {
                        __half2* tile = xrow + ((i & ~127) >> 1);
                        tile[kperm_pos(i & 127) >> 1] = __floats2half2_rn(xv[q][0] * mult, xv[q][1] * mult);
                        tile[kperm_pos((i & 127) + 2) >> 1] = __floats2half2_rn(xv[q][2] * mult, xv[q][3] * mult);
                    }
                }
                if (threadIdx.x == 0) xinv[t] = 1.0f / mult;
                __syncthreads();
            }
        };
        __syncthreads();   // the logits are in shared memory
        if (warp < T) topk_warp<false>(lg + warp * 256, E, k, sel + warp * 8, wsel + warp * 8, b == 0 ? a0.status : nullptr);
        __syncthreads();
        if (T == 1) {
            if (threadIdx.x < k) {
                const int j = threadIdx.x;
                act[j] = sel[j];
                act_np[j] = 1;
                act_pairs[j * 2] = Pair{0, j};
                cmap[j] = (j + 1) * 4;
                if (j == 0) *nact = k;
            }
        } else if (warp == 0) {
            const int n = T * k;
            const int t = lane / k, j = lane - (lane / k) * k;
            const int e = lane < n ? sel[t * 8 + j] : -1 - lane;
            int first = lane, p = 0;
            for (int i = 0; i < n; ++i) {
                const int ei = __shfl_sync(0xffffffffu, e, i);
                if (i < lane && ei == e) {
                    if (first == lane) first = i;
                    ++p;
                }
            }
            const uint32_t firsts = __ballot_sync(0xffffffffu, lane < n && first == lane);
            const int q = __popc(firsts & ((1u << first) - 1u));
            const uint32_t same = __match_any_sync(0xffffffffu, e);
            if (lane < n) {
                if (first == lane) {
                    act[q] = e;
                    act_np[q] = __popc(same);
                }
                act_pairs[q * 2 + p] = Pair{t, j};
                cmap[t * 8 + j] = (q + 1) * 4 + p;
            }
            if (lane == 0) *nact = __popc(firsts);
        }
        __syncthreads();
        const int na = *nact;
        const int n_units = na * units_per_expert;
        const int n_rs = a0.n_slots - 1;
        bool shared_pending = has_shared, wave_issued = false, x_staged = false;
        for (int u0 = b;;) {
            if (!wave_issued && u0 < n_units && ok) {
                __syncthreads();   // the previous wave's slots have been read
                if (threadIdx.x == 0) {
                    fence_proxy_async_smem();
#pragma unroll 1
                    for (int s2 = 0; s2 < n_rs; ++s2) {
                        const int u = u0 + s2 * G;
                        if (u < n_units) {
                            issue_half<WFMT>(al, act[u / units_per_expert], u % units_per_expert,
                                             slots + (size_t)s2 * al.unit_bytes, bars + s2);
                            mark_issued(s2);
                        }
                    }
                }
                wave_issued = true;
            }
            if (!x_staged) {
                stage_x();
                x_staged = true;
            }
            UnitRef wave[kMaxWaveUnits];
            int nw = 0;
            if (shared_pending) {
                wait_bar(shared_slot);
                wave[nw++] = UnitRef{slots + (size_t)shared_slot * al.unit_bytes, E, shared_unit, shared_pairs, T};
                shared_pending = false;
            } else if (u0 < n_units) {
#pragma unroll 1
                for (int s2 = 0; s2 < n_rs; ++s2) {
                    const int u = u0 + s2 * G;
                    if (u >= n_units) break;
                    wait_bar(s2);
                    const int q = u / units_per_expert;
                    wave[nw++] = UnitRef{slots + (size_t)s2 * al.unit_bytes, act[q], u % units_per_expert,
                                         act_pairs + q * 2, act_np[q]};
                }
                u0 += G * n_rs;
                wave_issued = false;
            } else {
                break;
            }
            if (ok && nw > 0) gateup_units<WFMT>(al, wave, nw, x16s, xinv, tss, acc);
        }
        // h is written: count this CTA in at the barrier, then, while the
        // barrier completes, request this CTA's routed down slabs (P2), the
        // next layer's shared half-unit (its slot is free now) and the next
        // layer's router slab (read in P2)
        if (ok) grid_arrive(gsync);
        if (threadIdx.x == 0 && ok) {
            fence_proxy_async_smem();
            if (down_tile >= 0 && na > 0) {
                mbar_arrive_expect_tx(bars + i_drouted, (uint32_t)(na * al.down_bytes));
#pragma unroll 1
                for (int q = 0; q < na; ++q)
                    issue_down<WFMT>(al, act[q], down_tile, down + (size_t)(1 + q) * al.down_bytes, bars + i_drouted);
                mark_issued(i_drouted);
            }
            if (!last) {
                const FusedArgs an = args_of(Ln);
                if (has_shared) {
                    issue_half<WFMT>(an, E, shared_unit, slots + (size_t)shared_slot * an.unit_bytes,
                                     bars + shared_slot);
                    mark_issued(shared_slot);
                }
                if (down_tile >= 0) {
                    mbar_arrive_expect_tx(bars + i_rslab, rslab_bytes);
                    bulk_g2s(rslab, Ln.router_t + (size_t)16 * down_tile * E, rslab_bytes, bars + i_rslab);
                    mark_issued(i_rslab);
                }
            }
        }
        if (ok && !grid_wait(gsync, a0.status)) ok = false;
        if (!ok) break;
        // ------------------------------------------------------------ P2
        if (last && b == 0) {   // every reader of this layer's accumulators has passed the barrier
            for (int i = threadIdx.x; i < kRaccCopies * T * E; i += kFThreads) {
                sa.racc[(size_t)buf * kRaccCopies * T * E + i] = 0ull;
                sa.rnf[(size_t)buf * kRaccCopies * T * E + i] = 0u;
            }
        }
        if (down_tile >= 0) {
            const int n_rows = T * (k + 1);
            const int nq = f >> 7;
            for (int r = warp; r < n_rows; r += kFWarps) {
                const float4* hr = reinterpret_cast<const float4*>(al.h + (size_t)r * f);
                float4 hv[8];
                float amax = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    hv[q] = q < nq ? __ldcg(hr + q * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(hv[q].x), fabsf(hv[q].y)), fmaxf(fabsf(hv[q].z), fabsf(hv[q].w))));
                }
                amax = warp_max(amax);
                const float mult = f16_range_mult(amax);
                __half2* hrow = reinterpret_cast<__half2*>(h16s + (size_t)r * f);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (q < nq) {
                        const int i = (q * 32 + lane) * 4;
                        __half2* tile = hrow + ((i & ~127) >> 1);
                        tile[kperm_pos(i & 127) >> 1] = __floats2half2_rn(hv[q].x * mult, hv[q].y * mult);
                        tile[kperm_pos((i & 127) + 2) >> 1] = __floats2half2_rn(hv[q].z * mult, hv[q].w * mult);
                    }
                }
                if (lane == 0) hinv[r] = 1.0f / mult;
            }
            wait_bar(i_dshared);
            if (na > 0) wait_bar(i_drouted);
            const int S = WFMT == 0 ? 64 : 128;
            const int kt_half = (KTf + 1) / 2;
#pragma unroll 1
            for (int it = warp; it < 2 * (na + 1) && ok; it += kFWarps) {
                const int q = it >> 1, hf = it & 1;
                const uint8_t* slab = down + (size_t)q * al.down_bytes;
                const uint8_t* cd = slab;
                const uint8_t* sd = slab + 2 * KTf * 512;
                const int np = q == 0 ? T : act_np[q - 1];
                const Pair* pp = q == 0 ? shared_pairs : act_pairs + (q - 1) * 2;
                const int hrow = g < np ? pp[g].t * (k + 1) + pp[g].j : -1;
                float cacc[4] = {0.f, 0.f, 0.f, 0.f};
                const int kt1 = min(KTf, (hf + 1) * kt_half);
#pragma unroll 1
                for (int kt = hf * kt_half; kt < kt1; ++kt) {
                    const uint4 wg = *reinterpret_cast<const uint4*>(cd + kt * 512 + lane * 16);
                    const uint4 wh = *reinterpret_cast<const uint4*>(cd + (KTf + kt) * 512 + lane * 16);
                    const TileScales<WFMT> sc = lds_scales<WFMT>(sd + kt * S, sd + (KTf + kt) * S, g);
                    uint32_t bfr[16];
                    if (hrow >= 0) {
                        lds_b16(h16s + (size_t)hrow * f + kt * 128 + c * 32, bfr);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) bfr[i] = 0u;
                    }
                    uint32_t fa[8][4];
                    decode_tile<WFMT>(wg, wh, sc, fa);
                    float sx[4][2];
                    if constexpr (WFMT == 1) block_sums_q41(bfr, sx);
                    mma_k128<WFMT>(cacc, fa, bfr, sc, sx);
                }
                float* dst = acc + (size_t)it * 128;
                dst[g * 8 + 2 * c] = cacc[0];
                dst[g * 8 + 2 * c + 1] = cacc[1];
                dst[(g + 8) * 8 + 2 * c] = cacc[2];
                dst[(g + 8) * 8 + 2 * c + 1] = cacc[3];
            }
            __syncthreads();
            // combine, residual in place: x[t][row] <- bf16(x + bf16(y_shared + sum_j w_j y_j))
            if (threadIdx.x < T * 16 && ok) {
                const int t = threadIdx.x / 16, rr = threadIdx.x % 16;
                const int orow = down_tile * 16 + rr;
                float v = (acc[rr * 8 + t] + acc[128 + rr * 8 + t]) * tss[E * 3 + 2] * hinv[t * (k + 1) + k];
                for (int j = 0; j < k; ++j) {
                    const int e = sel[t * 8 + j];
                    const int qp = cmap[t * 8 + j];
                    const float* aq = acc + (size_t)(qp >> 2) * 256 + rr * 8 + (qp & 3);
                    const float y = aq[0] + aq[128];
                    v += wsel[t * 8 + j] * (y * tss[e * 3 + 2] * hinv[t * (k + 1) + j]);
                }
                const __nv_bfloat16 o = __float2bfloat16_rn(v);
                const float r = __bfloat162float(__ldcg(sa.x + (size_t)t * d + orow));
                const __nv_bfloat16 xn = __float2bfloat16_rn(r + __bfloat162float(o));
                sa.x[(size_t)t * d + orow] = xn;
                xr[t * 16 + rr] = __bfloat162float(xn);
            }
            __syncthreads();   // down slabs read; xr written
            if (!last) {
                if (threadIdx.x == 0 && ok) {   // the next layer's shared down slab (slot 0 is free)
                    fence_proxy_async_smem();
                    const FusedArgs an = args_of(Ln);
                    mbar_arrive_expect_tx(bars + i_dshared, (uint32_t)an.down_bytes);
                    issue_down<WFMT>(an, E, down_tile, down, bars + i_dshared);
                    mark_issued(i_dshared);
                }
                wait_bar(i_rslab);
                if (ok) router_partials<T>(sa, rslab, xr, buf ^ 1, down_tile % kRaccCopies);
            }
        }
        if (!last && ok && !grid_sync(gsync, a0.status)) ok = false;
        Lc = Ln;
        Ln = Lnn;
    }
    drain();
}

}  // namespace

// Shared-memory plan of the fused kernel; 0 if it does not fit.
size_t fused_smem_bytes(const Shape& s, int T, int n_sms, int* n_slots_out, int offs[10]) {
    if (T < 1 || T > kFusedMaxT || s.n_shared != 1 || s.k > 8 || s.E > 256) return 0;
    if (s.d > 8 * kFThreads || s.f > 32 * 32) return 0;   // register staging of x and h rows
    const int S = s.wfmt == 0 ? 64 : 128;
    const int KTd = s.d / 128, KTf = s.f / 128;
    const size_t unit = (size_t)2 * KTd * (512 + S);   // one 8-row half-unit of gate and up
    const size_t dslab = (size_t)2 * KTf * (512 + S);
    const int max_active = T * s.k;
    const int units = max_active * (s.f / 8);
    if ((size_t)2 * s.d * 4 > unit) return 0;
    if ((s.E + n_sms - 1) / n_sms > 2) return 0;
    if (s.d / 16 > n_sms || s.f / 8 > n_sms) return 0;
    const size_t red = (size_t)kMaxWaveUnits * kFWarps * 128 * 4;
    const size_t accb = (size_t)(max_active + 1) * 2 * 128 * 4;
    int n_rs = (units + n_sms - 1) / n_sms;                 // routed slots for one wave
    if (n_rs > 3) n_rs = 3;
    size_t off = 0;
    auto take = [&](size_t n) { size_t o = off; off = (off + n + 127) / 128 * 128; return o; };
    for (;; --n_rs) {
        if (n_rs < 1) return 0;
        off = 0;
        offs[0] = (int)take((size_t)(n_rs + 1) * unit);     // + the shared expert's unit
        offs[1] = (int)unit;
        offs[2] = (int)take((size_t)(max_active + 1) * dslab);
        offs[3] = (int)dslab;
        offs[4] = (int)take(red > accb ? red : accb);
        offs[5] = (int)take((size_t)T * s.d * 2);
        offs[6] = (int)take((size_t)T * (s.k + 1) * s.f * 2);
        offs[7] = (int)take(4096);
        offs[8] = (int)take((size_t)T * s.d * 2);
        offs[9] = (int)take(tscale_bytes(s));
        if (off <= kFusedDynSmemMax) break;
    }
    *n_slots_out = n_rs + 1;
    return off;
}

cudaError_t prepare_decode_fused() {
    void (*kerns[4])(FusedArgs) = {decode_fused_kernel<0, 1>, decode_fused_kernel<0, 2>, decode_fused_kernel<1, 1>,
                                   decode_fused_kernel<1, 2>};
    void (*skerns[4])(StackArgs) = {decode_stack_kernel<0, 1>, decode_stack_kernel<0, 2>, decode_stack_kernel<1, 1>,
                                    decode_stack_kernel<1, 2>};
    auto opt_in = [](const void* kern) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e == cudaSuccess && fa.sharedSizeBytes + kFusedDynSmemMax > kMaxSmemOptin) e = cudaErrorInvalidValue;
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedDynSmemMax);
        if (e != cudaSuccess) cudaGetLastError();   // leave no error behind for later launch checks
        return e;
    };
    for (auto kern : kerns) {
        const cudaError_t e = opt_in(reinterpret_cast<const void*>(kern));
        if (e != cudaSuccess) return e;
    }
    for (auto kern : skerns) {
        const cudaError_t e = opt_in(reinterpret_cast<const void*>(kern));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The stack kernel's plan: the single-layer plan plus the router slab.
static size_t stack_plan(const Shape& s, int T, int n_sms, int* n_slots, int offs[10], int* off_rslab) {
    const size_t base = fused_smem_bytes(s, T, n_sms, n_slots, offs);
    if (base == 0 || s.d / 16 > n_sms) return 0;
    const size_t off = (base + 127) / 128 * 128;
    const size_t total = off + (size_t)16 * s.E * 4;
    if (total > kFusedDynSmemMax) return 0;
    *off_rslab = (int)off;
    return total;
}

size_t stack_smem_bytes(const Shape& s, int T, int n_sms) {
    int n_slots = 0, offs[10], off_rslab = 0;
    return stack_plan(s, T, n_sms, &n_slots, offs, &off_rslab);
}

namespace {
__global__ void transpose_router_kernel(const float* __restrict__ w, float* __restrict__ wt, int E, int d) {
    const long n = (long)E * d;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int e = (int)(i / d), j = (int)(i % d);
        wt[(size_t)j * E + e] = w[i];
    }
}
}  // namespace

cudaError_t transpose_router(const float* w, float* wt, int E, int d, cudaStream_t st) {
    transpose_router_kernel<<<148 * 4, 256, 0, st>>>(w, wt, E, d);
    return cudaGetLastError();
}

cudaError_t launch_decode_stack(const Shape& s, const StackLayer* layers_dev, int n_layers, __nv_bfloat16* x, int T,
                                const FusedScratch& fs, unsigned long long* gbar8, unsigned long long* racc,
                                uint32_t* rnf, int n_sms, cudaStream_t st) {
    int n_slots = 0, offs[10], off_rslab = 0;
    const size_t smem = stack_plan(s, T, n_sms, &n_slots, offs, &off_rslab);
    if (smem == 0 || n_layers < 1 || T < 1 || T > kFusedMaxT) return cudaErrorInvalidValue;
    StackArgs sa;
    FusedArgs& a = sa.f;
    a = FusedArgs{};
    a.cpm = s.codes_per_matrix();
    a.spm = s.scales_per_matrix();
    a.T = T;
    a.d = s.d;
    a.f = s.f;
    a.E = s.E;
    a.k = s.k;
    a.logits = fs.logits;
    a.h = fs.h;
    a.bar_count = reinterpret_cast<unsigned long long*>(fs.bar);
    a.status = fs.status;
    a.n_slots = n_slots;
    a.off_slots = offs[0];
    a.unit_bytes = offs[1];
    a.off_down = offs[2];
    a.down_bytes = offs[3];
    a.off_acc = offs[4];
    a.off_x16 = offs[5];
    a.off_h16 = offs[6];
    a.off_misc = offs[7];
    a.off_xbf = offs[8];
    a.off_ts = offs[9];
    a.ts_bytes = (int)tscale_bytes(s);
    sa.layers = layers_dev;
    sa.n = n_layers;
    sa.x = x;
    sa.gbar8 = gbar8;
    sa.racc = racc;
    sa.rnf = rnf;
    sa.off_rslab = off_rslab;
    void (*kern)(StackArgs) = s.wfmt == 0 ? (T == 1 ? decode_stack_kernel<0, 1> : decode_stack_kernel<0, 2>)
                                          : (T == 1 ? decode_stack_kernel<1, 1> : decode_stack_kernel<1, 2>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_sms);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, sa);
}

cudaError_t launch_decode_fused(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                                __nv_bfloat16* out, const __nv_bfloat16* residual, const FusedScratch& fs,
                                int n_sms, cudaStream_t st, const LayerDev* next) {
    int n_slots = 0, offs[10];
    const size_t smem = fused_smem_bytes(s, T, n_sms, &n_slots, offs);
    if (smem == 0) return cudaErrorInvalidValue;
    FusedArgs a;
    a.codes = L.codes;
    a.scales = L.scales;
    a.tscale = L.tscale;
    a.router = L.router;
    a.bias = L.bias;
    a.cpm = s.codes_per_matrix();
    a.spm = s.scales_per_matrix();
    a.x = x;
    a.out = out;
    a.residual = residual;
    a.T = T;
    a.d = s.d;
    a.f = s.f;
    a.E = s.E;
    a.k = s.k;
    a.logits = fs.logits;
    a.h = fs.h;
    a.bar_count = reinterpret_cast<unsigned long long*>(fs.bar);
    a.status = fs.status;
    a.n_slots = n_slots;
    a.off_slots = offs[0];
    a.unit_bytes = offs[1];
    a.off_down = offs[2];
    a.down_bytes = offs[3];
    a.off_acc = offs[4];
    a.off_x16 = offs[5];
    a.off_h16 = offs[6];
    a.off_misc = offs[7];
    a.off_xbf = offs[8];
    a.off_ts = offs[9];
    a.ts_bytes = (int)tscale_bytes(s);
    a.next_codes = next != nullptr ? next->codes : nullptr;
    a.next_scales = next != nullptr ? next->scales : nullptr;
    a.next_router = next != nullptr ? next->router : nullptr;
    void (*kern)(FusedArgs) = s.wfmt == 0 ? (T == 1 ? decode_fused_kernel<0, 1> : decode_fused_kernel<0, 2>)
                                          : (T == 1 ? decode_fused_kernel<1, 1> : decode_fused_kernel<1, 2>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_sms);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace flint
