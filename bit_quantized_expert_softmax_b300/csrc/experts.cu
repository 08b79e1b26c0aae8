// Expert projections for small and medium token counts: SwiGLU gate/up,
// down projection and the weighted combine with the shared expert.
//
// The Flint blog ("Recursive Flint 40B-A2.5B", section "The architecture is
// an argument about memory bandwidth") frames decode as moving the selected
// experts' weights from memory to the arithmetic units; these kernels stream
// only the selected experts' packed 4-bit tiles, once, with one 16-byte load
// per lane per 8x128 tile, and decode them in registers.
//
// Arithmetic: activations are fp16 scaled per token (or per position) by a
// power of two that brings their maximum into [2^14, 2^15), and mma.sync
// m16n8k16 accumulates in fp32. NVFP4 weights enter the MMA as E2M1 x E4M3
// (exact in fp16) and their fp32 tensor scale is applied to the accumulator.
// q4_1 weights enter as their codes q (exact); per 32-element block the
// accumulator takes d * sum(q x) + m * sum(x), so d*q + m is never rounded
// (tiles.cuh, mma_k128). The inverse activation scale is applied last.
#include <cstdlib>

#include "kernels.cuh"
#include "pdl.cuh"
#include "tiles.cuh"
#include "umma.cuh"

namespace flint {

namespace {

constexpr int kThreads = 128;   // 4 warps
constexpr int kNB = 4;          // n-tiles (8 tokens each) per pass

struct ExpertArgs {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* tscale;
    size_t codes_per_mat, scales_per_mat;
    int d, f, E, k, n_shared, T;
    Workspace ws;
    __nv_bfloat16* out;
    const __nv_bfloat16* residual;
    int fuse_combine;
};

__device__ __forceinline__ int token_of(const ExpertArgs& a, int pos) {
    const int routed = a.T * a.k;
    return pos < routed ? __ldg(a.ws.perm + pos) / a.k : pos - routed;
}

// ---------------------------------------------------------------------------
// a5 + a7 (gate/up part): h = silu(W_gate x) * (W_up x) for one 16-row tile of
// f for every position of one active expert slot.
// ---------------------------------------------------------------------------
template <int WFMT>
__global__ void __launch_bounds__(kThreads) gateup_kernel(ExpertArgs a) {
    griddep_wait();
    __shared__ float red[4][2][kNB][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KT = a.d >> 7;
    const int tiles = a.f >> 4;
    // a task is (slot, 16-row tile, pass of 8*kNB positions), the pass
    // innermost: the passes of a slot with many positions run on different
    // CTAs at once instead of one after another (a pass beyond the slot's
    // positions is empty)
    const int max_pass = (a.T + 8 * kNB - 1) / (8 * kNB);
    const int n_tasks = a.ws.meta[0] * tiles * max_pass;
    const size_t tile_bytes_s = (WFMT == 0) ? 64 : 128;
    for (int task = blockIdx.x; task < n_tasks; task += gridDim.x) {
        const int pass = task % max_pass, rest = task / max_pass;
        const int slot = rest / tiles, r16 = rest - slot * tiles;
        const int e = a.ws.slot_expert[slot];
        const int p0 = a.ws.slot_off[slot], cnt = a.ws.slot_cnt[slot];
        const uint8_t* cbase = a.codes + (size_t)e * 3 * a.codes_per_mat;
        const uint8_t* sbase = a.scales + (size_t)e * 3 * a.scales_per_mat;
        const float tsg = a.tscale[e * 3 + 0], tsu = a.tscale[e * 3 + 1];
        const size_t rtg = (size_t)(2 * r16) * KT, rth = (size_t)(2 * r16 + 1) * KT;
        for (int n0 = pass * 8 * kNB; n0 < cnt && n0 < (pass + 1) * 8 * kNB; n0 += 8 * kNB) {
            const int nb = min(kNB, (cnt - n0 + 7) >> 3);
            float accg[kNB][4], accu[kNB][4];
#pragma unroll
            for (int i = 0; i < kNB; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) accg[i][j] = accu[i][j] = 0.f;
            int tok[kNB];
#pragma unroll
            for (int nt = 0; nt < kNB; ++nt) {
                const int n = n0 + nt * 8 + g;
                tok[nt] = (nt < nb && n < cnt) ? token_of(a, p0 + n) : -1;
            }
            for (int kt = warp; kt < KT; kt += 4) {
                const uint8_t* cg = cbase;                       // gate
                const uint8_t* cu = cbase + a.codes_per_mat;     // up
                const uint4 wgg = ldg_nc_v4(cg + (rtg + kt) * 512 + lane * 16);
                const uint4 wgh = ldg_nc_v4(cg + (rth + kt) * 512 + lane * 16);
                const uint4 wug = ldg_nc_v4(cu + (rtg + kt) * 512 + lane * 16);
                const uint4 wuh = ldg_nc_v4(cu + (rth + kt) * 512 + lane * 16);
                const uint8_t* sg = sbase;
                const uint8_t* su = sbase + a.scales_per_mat;
                const TileScales<WFMT> scg = load_scales<WFMT>(sg + (rtg + kt) * tile_bytes_s,
                                                               sg + (rth + kt) * tile_bytes_s, g);
                const TileScales<WFMT> scu = load_scales<WFMT>(su + (rtg + kt) * tile_bytes_s,
                                                               su + (rth + kt) * tile_bytes_s, g);
                uint32_t fa[8][4], fu[8][4];
                decode_tile<WFMT>(wgg, wgh, scg, fa);
                decode_tile<WFMT>(wug, wuh, scu, fu);
#pragma unroll
                for (int nt = 0; nt < kNB; ++nt) {
                    if (nt >= nb) break;
                    uint32_t b[16];
                    if (tok[nt] >= 0) {
                        const uint4* xp = reinterpret_cast<const uint4*>(
                            a.ws.x16 + (size_t)tok[nt] * a.d + kt * 128 + c * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v = __ldg(xp + q);
                            b[4 * q + 0] = v.x;
                            b[4 * q + 1] = v.y;
                            b[4 * q + 2] = v.z;
                            b[4 * q + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) b[q] = 0u;
                    }
                    float sx[4][2];
                    if constexpr (WFMT == 1) block_sums_q41(b, sx);
                    mma_k128<WFMT>(accg[nt], fa, b, scg, sx);
                    mma_k128<WFMT>(accu[nt], fu, b, scu, sx);
                }
            }
            // reduce the four K-partials
#pragma unroll
            for (int nt = 0; nt < kNB; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    red[warp][0][nt][lane][j] = accg[nt][j];
                    red[warp][1][nt][lane][j] = accu[nt][j];
                }
            __syncthreads();
            const int nt = warp;
            if (nt < nb) {
                float hv[4];
                int posv[2] = {-1, -1};
                float xinv[2] = {0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = n0 + nt * 8 + 2 * c + q;
                    if (n < cnt) {
                        posv[q] = p0 + n;
                        xinv[q] = a.ws.xinv[token_of(a, p0 + n)];
                    }
                }
                float hmax[2] = {0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float sg = ((red[0][0][nt][lane][j] + red[1][0][nt][lane][j]) +
                                      red[2][0][nt][lane][j]) + red[3][0][nt][lane][j];
                    const float su = ((red[0][1][nt][lane][j] + red[1][1][nt][lane][j]) +
                                      red[2][1][nt][lane][j]) + red[3][1][nt][lane][j];
                    const int q = j & 1;
                    const float gv = sg * tsg * xinv[q];
                    const float uv = su * tsu * xinv[q];
                    hv[j] = gv / (1.0f + expf(-gv)) * uv;
                    if (posv[q] >= 0) hmax[q] = fmaxf(hmax[q], fabsf(hv[j]));
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int q = j & 1;
                    if (posv[q] < 0) continue;
                    const int row = r16 * 16 + g + ((j >> 1) << 3);
                    a.ws.hf[(size_t)posv[q] * a.f + (row & ~127) + kperm_pos(row & 127)] = hv[j];
                }
                // max over the 8 row groups sharing these positions
#pragma unroll
                for (int q = 0; q < 2; ++q) {
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1)
                        hmax[q] = fmaxf(hmax[q], __shfl_xor_sync(0xffffffffu, hmax[q], o));
                }
                if (g == 0) {
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        if (posv[q] >= 0) atomicMax(a.ws.hamax + posv[q], __float_as_uint(hmax[q]));
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// a6 + a7 + a8: y = W_down h for 64 output rows of one active slot, weighted
// by the routing weight (1 for the shared expert) into yw; with fuse_combine,
// the last slot to finish a row block sums the block's outputs in slot order
// and writes bf16.
// ---------------------------------------------------------------------------
__device__ void combine_rows(const ExpertArgs& a, int row0, int nrows) {
    const int T = a.T;
    for (int i = threadIdx.x; i < T * nrows; i += blockDim.x) {
        const int t = i / nrows, row = row0 + i % nrows;
        float v = 0.f;
        if (a.n_shared) v = __ldcg(a.ws.yw + (size_t)(T * a.k + t) * a.d + row);
        for (int j = 0; j < a.k; ++j) {
            const int pos = __ldcg(a.ws.inv + t * a.k + j);
            v += __ldcg(a.ws.yw + (size_t)pos * a.d + row);
        }
        __nv_bfloat16 o = __float2bfloat16_rn(v);
        if (a.residual != nullptr) {
            const float r = __bfloat162float(a.residual[(size_t)t * a.d + row]);
            o = __float2bfloat16_rn(r + __bfloat162float(o));
        }
        a.out[(size_t)t * a.d + row] = o;
    }
}

// Per pass of up to kDownPos positions the CTA stages their h (already
// fragment-permuted by the gate/up kernel) once in shared memory as fp16,
// k-chunk by k-chunk, instead of every warp reading it from L2 per k-tile;
// each warp's weight loads for the chunk are issued before the staging so
// that the DRAM and L2 round trips overlap.
constexpr int kDownPos = 8 * kNB;   // positions per pass
constexpr int kDownKC = 4;          // k-tiles per staged chunk
static_assert(kDownPos >= kFuseCombineT, "the fused combine counts one arrival per (slot, block)");

template <int WFMT>
__global__ void __launch_bounds__(kThreads) down_kernel(ExpertArgs a) {
    griddep_wait();
    __shared__ __align__(16) __half hs[kDownPos * kDownKC * 128];   // [position][chunk K], fp16
    __shared__ float hmul[kDownPos];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KT = a.f >> 7;
    const int blocks = a.d >> 6;
    const int n_slots = a.ws.meta[0];
    // task = (slot, 64-row block, pass of kDownPos positions), pass innermost
    // (with the fused combine, T <= kFuseCombineT gives one pass per slot, so
    // each (slot, block) task still arrives exactly once)
    const int max_pass = (a.T + kDownPos - 1) / kDownPos;
    const int n_tasks = n_slots * blocks * max_pass;
    const size_t tile_bytes_s = (WFMT == 0) ? 64 : 128;
    constexpr int kRow = kDownKC * 128;   // staged halves per position
    for (int task = blockIdx.x; task < n_tasks; task += gridDim.x) {
        const int pass = task % max_pass, rest = task / max_pass;
        const int blk = rest % blocks, slot = rest / blocks;
        const int e = a.ws.slot_expert[slot];
        const int p0 = a.ws.slot_off[slot], cnt = a.ws.slot_cnt[slot];
        const bool shared = (e == a.E);
        const uint8_t* cd = a.codes + ((size_t)e * 3 + 2) * a.codes_per_mat;
        const uint8_t* sd = a.scales + ((size_t)e * 3 + 2) * a.scales_per_mat;
        const float tsd = a.tscale[e * 3 + 2];
        const int r16 = blk * 4 + warp;
        const size_t rtg = (size_t)(2 * r16) * KT, rth = (size_t)(2 * r16 + 1) * KT;
        for (int n0 = pass * kDownPos; n0 < cnt && n0 < (pass + 1) * kDownPos; n0 += kDownPos) {
            const int np = min(kDownPos, cnt - n0);
            const int nb = (np + 7) >> 3;
            float acc[kNB][4];
#pragma unroll
            for (int i = 0; i < kNB; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
            __syncthreads();   // the previous pass is done with hs and hmul
            if (threadIdx.x < np) hmul[threadIdx.x] = f16_range_mult(__uint_as_float(a.ws.hamax[p0 + n0 + threadIdx.x]));
            for (int kc = 0; kc < KT; kc += kDownKC) {
                const int nkc = min(kDownKC, KT - kc);
                uint4 wg[kDownKC], wh[kDownKC];
                TileScales<WFMT> sc[kDownKC];
#pragma unroll
                for (int i = 0; i < kDownKC; ++i) {
                    if (i < nkc) {
                        wg[i] = ldg_nc_v4(cd + (rtg + kc + i) * 512 + lane * 16);
                        wh[i] = ldg_nc_v4(cd + (rth + kc + i) * 512 + lane * 16);
                        sc[i] = load_scales<WFMT>(sd + (rtg + kc + i) * tile_bytes_s, sd + (rth + kc + i) * tile_bytes_s,
                                                  g);
                    }
                }
                __syncthreads();   // hmul written; the previous chunk's reads of hs are done
                const int row_f4 = nkc * 32;   // float4 of one position in this chunk
                for (int i = threadIdx.x; i < np * row_f4; i += kThreads) {
                    const int pl = i / row_f4, q = i - pl * row_f4;
                    const float4 v = __ldcg(
                        reinterpret_cast<const float4*>(a.ws.hf + (size_t)(p0 + n0 + pl) * a.f + kc * 128) + q);
                    const float m = hmul[pl];
                    *reinterpret_cast<uint2*>(hs + pl * kRow + q * 4) =
                        make_uint2(pack_half2(v.x * m, v.y * m), pack_half2(v.z * m, v.w * m));
                }
                __syncthreads();
                for (int i = 0; i < nkc; ++i) {
                    uint32_t fa[8][4];
                    decode_tile<WFMT>(wg[i], wh[i], sc[i], fa);
#pragma unroll
                    for (int nt = 0; nt < kNB; ++nt) {
                        if (nt >= nb) break;
                        const int pl = nt * 8 + g;
                        uint32_t b[16];
                        if (pl < np) {
                            const uint4* hp = reinterpret_cast<const uint4*>(hs + pl * kRow + i * 128 + c * 32);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint4 v = hp[q];
                                b[4 * q + 0] = v.x;
                                b[4 * q + 1] = v.y;
                                b[4 * q + 2] = v.z;
                                b[4 * q + 3] = v.w;
                            }
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; ++q) b[q] = 0u;
                        }
                        float sx[4][2];
                        if constexpr (WFMT == 1) block_sums_q41(b, sx);
                        mma_k128<WFMT>(acc[nt], fa, b, sc[i], sx);
                    }
                }
            }
            // epilogue: rows g, g+8 of this warp's tile; positions 2c, 2c+1 of each n-tile
#pragma unroll
            for (int nt = 0; nt < kNB; ++nt) {
                if (nt >= nb) break;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = n0 + nt * 8 + 2 * c + q;
                    if (n >= cnt) continue;
                    const int pos = p0 + n;
                    const float wr = shared ? 1.0f : a.ws.w[__ldg(a.ws.perm + pos)];
                    const float mult = f16_range_mult(__uint_as_float(a.ws.hamax[pos]));
                    const float sc_ = tsd / mult * wr;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int row = r16 * 16 + g + hh * 8;
                        a.ws.yw[(size_t)pos * a.d + row] = acc[nt][hh * 2 + q] * sc_;
                    }
                }
            }
        }
        if (a.fuse_combine) {
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                const uint32_t prev = atomicAdd(a.ws.counters + 1 + blk, 1u);
                s_last = (prev == (uint32_t)n_slots - 1u);
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                combine_rows(a, blk * 64, 64);
                if (threadIdx.x == 0) a.ws.counters[1 + blk] = 0u;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Ring-fed variants (T <= kSmallT): persistent CTAs, two per SM, whose tasks'
// weights arrive in shared memory by 1-D bulk copies several tasks ahead,
// instead of each warp holding one k-tile of loads in flight. A task's
// weights are contiguous in the tile layout (the tile rows of a row range
// follow each other, k-tiles innermost), so a task is four copies (gate/up)
// or two (down). A task is (slot, row unit, pass of 8 kNB positions); thread
// 0 takes the next task from a global counter when it issues a fill, so that
// CTAs which drew cheap tasks (few positions) take more of them, and records
// it for the stage's consumers. The last CTA to leave resets the counter.
// ---------------------------------------------------------------------------
constexpr int kRingWarps = 4;
constexpr int kRingThreads = 32 * kRingWarps;
constexpr int kRingMaxStages = 4;
// two CTAs per SM: while one is in its barriers and epilogue the other computes
constexpr int kRingCtasPerSm = 2;
constexpr int kRingSmemCap = 112 * 1024;
constexpr int kRingMaxSlots = 512;                // task table entries (active slots; E <= 256)
constexpr int kRingCtr = kCounters - 64;          // [0, 1]: gate/up task and exit counters; [2, 3]: down
static_assert(kRingCtr > 1 + 4096 / 64 && kRingCtr + 4 <= kCounters - kSmallT / 8, "counter ranges overlap");

__host__ __device__ __forceinline__ int scale_tile_bytes(int wfmt) { return wfmt == 0 ? 64 : 128; }

// gate/up task: 16 rows of f (two tile rows) of gate and of up, full K
__host__ __device__ __forceinline__ uint32_t gu_stage_bytes(int KT, int wfmt) {
    return 4u * (uint32_t)KT * (512u + (uint32_t)scale_tile_bytes(wfmt));
}
constexpr int kGuRedBytes = kRingWarps * 2 * kNB * 32 * 4 * 4;   // the warps' K-partials of gate and up

// down task: 16 output rows per warp (two tile rows each), full K
constexpr int kDnRows = 16 * kRingWarps;
constexpr int kDnChunk = 2;   // consecutive down tasks (row blocks of one pass) a CTA takes at once
__host__ __device__ __forceinline__ uint32_t dn_stage_bytes(int KTf, int wfmt) {
    return 2u * kRingWarps * (uint32_t)KTf * (512u + (uint32_t)scale_tile_bytes(wfmt));
}
// staged h rows: f fp16 + 8 of padding, so that the fragment reads of the
// 8 positions of an n-tile (rows otherwise a multiple of 128 bytes apart) fall
// in distinct banks
__host__ __device__ __forceinline__ int dn_hs_pitch(int f) { return f + 8; }
__host__ __device__ __forceinline__ uint32_t dn_hs_bytes(int f) { return (uint32_t)kDownPos * dn_hs_pitch(f) * 2; }

// shared memory in front of the ring: barriers and task records, then the
// task table, then the kernel's own buffer
struct RingHead {
    uint64_t full[kRingMaxStages];
    int4 task[kRingMaxStages];        // slot (-1: no task), unit, pass, -
    int wsum[kRingWarps];
    int n_tasks;
    int pre[kRingMaxSlots + 1];       // the slot of rank r owns tasks [pre[r], pre[r + 1])
    int ord[kRingMaxSlots];           // rank -> slot
    int cnt[kRingMaxSlots];           // positions of each slot
};
constexpr uint32_t kRingHeadBytes = (sizeof(RingHead) + 127) / 128 * 128;

struct RingLayout {
    int stages;
    uint32_t stage_bytes, extra_bytes, smem;
};

// extra_bytes: everything in front of the ring
__host__ __forceinline__ RingLayout ring_layout(uint32_t stage_bytes, uint32_t extra_bytes) {
    RingLayout r{0, stage_bytes, extra_bytes, 0};
    int s = kRingMaxStages;
    while (s >= 2 && extra_bytes + s * stage_bytes > (uint32_t)kRingSmemCap) --s;
    r.stages = s >= 2 ? s : 0;
    r.smem = extra_bytes + (uint32_t)r.stages * stage_bytes;
    return r;
}
__host__ __forceinline__ RingLayout gu_layout(const Shape& s) {
    return ring_layout(gu_stage_bytes(s.d >> 7, s.wfmt), kRingHeadBytes + kGuRedBytes);
}
__host__ __forceinline__ RingLayout dn_layout(const Shape& s) {
    return ring_layout(dn_stage_bytes(s.f >> 7, s.wfmt), kRingHeadBytes + kDownPos * 4 + dn_hs_bytes(s.f));
}

// The task table. Slots are ranked by their number of positions, most first
// (ties: lower slot first), so that the tasks of full passes -- the shared
// expert's and the popular experts' -- are handed out before the short ones
// and the last tasks to start are the cheapest. Every CTA computes the same
// table. Then every thread takes consecutive ranks, one block scan.
// units: row units per pass of a slot. Returns the number of tasks.
__device__ int ring_task_table(const ExpertArgs& a, int units, RingHead* hd) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ns = min(a.ws.meta[0], kRingMaxSlots);
    for (int sl = threadIdx.x; sl < ns; sl += kRingThreads) hd->cnt[sl] = a.ws.slot_cnt[sl];
    __syncthreads();
    for (int sl = threadIdx.x; sl < ns; sl += kRingThreads) {
        const int c = hd->cnt[sl];
        int r = 0;
        for (int j = 0; j < ns; ++j) {
            const int cj = hd->cnt[j];
            r += (cj > c || (cj == c && j < sl)) ? 1 : 0;
        }
        hd->ord[r] = sl;
    }
    __syncthreads();
    const int per = (ns + kRingThreads - 1) / kRingThreads;
    const int s0 = threadIdx.x * per;
    int mine[kRingMaxSlots / kRingThreads];
    int local = 0;
#pragma unroll
    for (int j = 0; j < kRingMaxSlots / kRingThreads; ++j) {
        const int sl = s0 + j;
        mine[j] = (j < per && sl < ns) ? units * ((hd->cnt[hd->ord[sl]] + 8 * kNB - 1) / (8 * kNB)) : 0;
        local += mine[j];
    }
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) hd->wsum[warp] = x;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kRingWarps; ++w) {
        if (w < warp) base += hd->wsum[w];
        total += hd->wsum[w];
    }
    int run = base + x - local;
#pragma unroll
    for (int j = 0; j < kRingMaxSlots / kRingThreads; ++j) {
        const int sl = s0 + j;
        if (j < per && sl < ns) hd->pre[sl] = run;
        run += mine[j];
    }
    if (threadIdx.x == 0) {
        hd->pre[ns] = total;
        hd->n_tasks = total;
    }
    __syncthreads();
    return total;
}

// task index -> (slot, unit, pass) by binary search in the table
__device__ __forceinline__ int4 ring_decode(const RingHead* hd, int ns, int units, int t) {
    int lo = 0, hi = ns;   // pre[lo] <= t < pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (hd->pre[mid] <= t) lo = mid; else hi = mid;
    }
    const int r = t - hd->pre[lo];
    return make_int4(hd->ord[lo], r % units, r / units, 0);
}

// Thread 0: fill number `fill` into stage fill % stages. Takes the next task
// of the chunk [next, end) it holds, or a new chunk of `chunk` consecutive
// tasks from the counter (unless the counter has run out before); with no
// task left, records slot -1 and completes the stage's phase with a plain
// arrival.
template <class Issue>
__device__ __forceinline__ void ring_fill(RingHead* hd, int stages, uint32_t fill, int ns, int units,
                                          unsigned* ctr, int chunk, int& next, int& end, bool& out, Issue issue) {
    const int s = (int)(fill % (uint32_t)stages);
    int t = -1;
    if (!out) {
        if (next >= end) {
            next = (int)atomicAdd(ctr, (unsigned)chunk);
            end = next + chunk;
        }
        t = next++;
        if (t >= hd->n_tasks) {
            t = -1;
            out = true;
        }
    }
    if (t < 0) {
        hd->task[s] = make_int4(-1, 0, 0, 0);
        mbar_arrive(&hd->full[s]);
    } else {
        const int4 tk = ring_decode(hd, ns, units, t);
        hd->task[s] = tk;
        issue(tk, s);
    }
}

// Wait (bounded) for the stage of fill i; all threads agree on the outcome.
__device__ __forceinline__ bool ring_acquire(uint64_t* full, int stages, int i, uint32_t* status) {
    const bool got = mbar_wait_bounded(&full[i % stages], (uint32_t)(i / stages) & 1u, status);
    return __syncthreads_and(got) != 0;
}

// Thread 0, on the way out: no copy of this CTA still in flight; the last CTA
// to leave resets the task and exit counters for the next launch.
__device__ __forceinline__ void ring_exit(RingHead* hd, int stages, uint32_t fills, unsigned* ctr, uint32_t* status) {
    drain_ring(hd->full, stages, fills, status);
    __threadfence();
    if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
        __threadfence();
        atomicExch(ctr, 0u);
        atomicExch(ctr + 1, 0u);
    }
}

// n-tile nt of a gate/up pass: sums the warps' K-partials (fixed order),
// h = silu(g) * u per (row, position), stores h fragment-permuted and raises
// the positions' max |h|.
__device__ __forceinline__ void gu_epilogue(const ExpertArgs& a, const float* red, int nt, int lane, int n0, int p0,
                                            int cnt, int r16, float tsg, float tsu) {
    const int g = lane >> 2, c = lane & 3;
    auto R = [&](int w, int m, int j) { return red[(((w * 2 + m) * kNB + nt) * 32 + lane) * 4 + j]; };
    int posv[2] = {-1, -1};
    float xinv[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int n = n0 + nt * 8 + 2 * c + q;
        if (n < cnt) {
            posv[q] = p0 + n;
            xinv[q] = a.ws.xinv[token_of(a, p0 + n)];
        }
    }
    float hv[4];
    float hmax[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float sg = R(0, 0, j), su = R(0, 1, j);
#pragma unroll
        for (int w = 1; w < kRingWarps; ++w) {
            sg += R(w, 0, j);
            su += R(w, 1, j);
        }
        const int q = j & 1;
        const float gv = sg * tsg * xinv[q];
        const float uv = su * tsu * xinv[q];
        hv[j] = gv / (1.0f + expf(-gv)) * uv;
        if (posv[q] >= 0) hmax[q] = fmaxf(hmax[q], fabsf(hv[j]));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int q = j & 1;
        if (posv[q] < 0) continue;
        const int row = r16 * 16 + g + ((j >> 1) << 3);
        a.ws.hf[(size_t)posv[q] * a.f + (row & ~127) + kperm_pos(row & 127)] = hv[j];
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) hmax[q] = fmaxf(hmax[q], __shfl_xor_sync(0xffffffffu, hmax[q], o));
    }
    if (g == 0) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (posv[q] >= 0) atomicMax(a.ws.hamax + posv[q], __float_as_uint(hmax[q]));
    }
}

template <int WFMT>
__device__ __forceinline__ void gu_issue(const ExpertArgs& a, int4 tk, int KT, uint8_t* st, uint64_t* bar) {
    const int e = __ldg(a.ws.slot_expert + tk.x);
    const uint32_t cb = 2u * KT * 512u, sb = 2u * KT * (uint32_t)scale_tile_bytes(WFMT);
    const uint8_t* cg = a.codes + (size_t)e * 3 * a.codes_per_mat + (size_t)tk.y * cb;
    const uint8_t* sg = a.scales + (size_t)e * 3 * a.scales_per_mat + (size_t)tk.y * sb;
    mbar_arrive_expect_tx(bar, 2 * cb + 2 * sb);
    bulk_g2s(st, cg, cb, bar);
    bulk_g2s(st + cb, cg + a.codes_per_mat, cb, bar);
    bulk_g2s(st + 2 * cb, sg, sb, bar);
    bulk_g2s(st + 2 * cb + sb, sg + a.scales_per_mat, sb, bar);
}

// a5 + a7 (gate/up part), task = (slot, 16 rows of f, pass of 8 kNB
// positions); the warps split K and their partials are summed in shared
// memory.
template <int WFMT>
__global__ void __launch_bounds__(kRingThreads, kRingCtasPerSm) gateup_ring_kernel(ExpertArgs a, int stages, uint32_t stage_bytes) {
    griddep_wait();
    extern __shared__ __align__(128) uint8_t rsm[];
    RingHead* hd = reinterpret_cast<RingHead*>(rsm);
    float* red = reinterpret_cast<float*>(rsm + kRingHeadBytes);    // [warps][2][kNB][32][4]
    uint8_t* ring = rsm + kRingHeadBytes + kGuRedBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KT = a.d >> 7;
    const int units = a.f >> 4;
    unsigned* ctr = a.ws.counters + kRingCtr;
    constexpr int TSB = (WFMT == 0) ? 64 : 128;
    const uint32_t cb = 2u * KT * 512u, sb = 2u * KT * TSB;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&hd->full[s], 1);
        mbar_fence_init();
    }
    ring_task_table(a, units, hd);   // (its barriers also publish the initialised mbarriers)
    const int ns = min(a.ws.meta[0], kRingMaxSlots);
    uint32_t fills = 0;
    bool out = false;
    int tnext = 0, tend = 0;   // one task per grab
    auto issue = [&](int4 tk, int s) {
        gu_issue<WFMT>(a, tk, KT, ring + s * stage_bytes, &hd->full[s]);
    };
    if (threadIdx.x == 0)
        for (; (int)fills < stages; ++fills) ring_fill(hd, stages, fills, ns, units, ctr, 1, tnext, tend, out, issue);
    auto R = [&](int w, int m, int nt, int j) -> float& { return red[(((w * 2 + m) * kNB + nt) * 32 + lane) * 4 + j]; };
    for (int i = 0;; ++i) {
        if (!ring_acquire(hd->full, stages, i, a.ws.status)) break;
        const int4 tk = hd->task[i % stages];
        if (tk.x < 0) break;
        const int slot = tk.x, r16 = tk.y, n0 = tk.z * 8 * kNB;
        const int e = a.ws.slot_expert[slot];
        const int p0 = a.ws.slot_off[slot], cnt = a.ws.slot_cnt[slot];
        const float tsg = a.tscale[e * 3 + 0], tsu = a.tscale[e * 3 + 1];
        const uint8_t* st = ring + (i % stages) * stage_bytes;
        const uint8_t* sgc = st;               // gate codes: tile rows 2 r16, 2 r16 + 1
        const uint8_t* suc = st + cb;          // up codes
        const uint8_t* sgs = st + 2 * cb;      // gate scales
        const uint8_t* sus = st + 2 * cb + sb; // up scales
        const int nb = min(kNB, (cnt - n0 + 7) >> 3);
        float accg[kNB][4], accu[kNB][4];
#pragma unroll
        for (int q = 0; q < kNB; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) accg[q][j] = accu[q][j] = 0.f;
        int tok[kNB];
#pragma unroll
        for (int nt = 0; nt < kNB; ++nt) {
            const int n = n0 + nt * 8 + g;
            tok[nt] = (nt < nb && n < cnt) ? token_of(a, p0 + n) : -1;
        }
        for (int kt = warp; kt < KT; kt += kRingWarps) {
            const uint4 wgg = *reinterpret_cast<const uint4*>(sgc + kt * 512 + lane * 16);
            const uint4 wgh = *reinterpret_cast<const uint4*>(sgc + (KT + kt) * 512 + lane * 16);
            const uint4 wug = *reinterpret_cast<const uint4*>(suc + kt * 512 + lane * 16);
            const uint4 wuh = *reinterpret_cast<const uint4*>(suc + (KT + kt) * 512 + lane * 16);
            const TileScales<WFMT> scg = lds_scales<WFMT>(sgs + kt * TSB, sgs + (KT + kt) * TSB, g);
            const TileScales<WFMT> scu = lds_scales<WFMT>(sus + kt * TSB, sus + (KT + kt) * TSB, g);
            uint32_t fa[8][4], fu[8][4];
            decode_tile<WFMT>(wgg, wgh, scg, fa);
            decode_tile<WFMT>(wug, wuh, scu, fu);
#pragma unroll
            for (int nt = 0; nt < kNB; ++nt) {
                if (nt >= nb) break;
                uint32_t b[16];
                if (tok[nt] >= 0) {
                    const uint4* xp = reinterpret_cast<const uint4*>(a.ws.x16 + (size_t)tok[nt] * a.d + kt * 128 + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 v = __ldg(xp + q);
                        b[4 * q + 0] = v.x;
                        b[4 * q + 1] = v.y;
                        b[4 * q + 2] = v.z;
                        b[4 * q + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) b[q] = 0u;
                }
                float sx[4][2];
                if constexpr (WFMT == 1) block_sums_q41(b, sx);
                mma_k128<WFMT>(accg[nt], fa, b, scg, sx);
                mma_k128<WFMT>(accu[nt], fu, b, scu, sx);
            }
        }
#pragma unroll
        for (int nt = 0; nt < kNB; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                R(warp, 0, nt, j) = accg[nt][j];
                R(warp, 1, nt, j) = accu[nt][j];
            }
        __syncthreads();   // partials written; every thread is done with the stage's weights
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            ring_fill(hd, stages, fills, ns, units, ctr, 1, tnext, tend, out, issue);
            ++fills;
        }
        if (warp < nb) gu_epilogue(a, red, warp, lane, n0, p0, cnt, r16, tsg, tsu);
        __syncthreads();   // partials read
    }
    if (threadIdx.x == 0) ring_exit(hd, stages, fills, ctr, a.ws.status);
}

template <int WFMT>
__device__ __forceinline__ void dn_issue(const ExpertArgs& a, int4 tk, int KTf, uint8_t* st, uint64_t* bar) {
    const int e = __ldg(a.ws.slot_expert + tk.x);
    const uint32_t cb = 2u * kRingWarps * KTf * 512u, sb = 2u * kRingWarps * KTf * (uint32_t)scale_tile_bytes(WFMT);
    mbar_arrive_expect_tx(bar, cb + sb);
    bulk_g2s(st, a.codes + ((size_t)e * 3 + 2) * a.codes_per_mat + (size_t)tk.y * cb, cb, bar);
    bulk_g2s(st + cb, a.scales + ((size_t)e * 3 + 2) * a.scales_per_mat + (size_t)tk.y * sb, sb, bar);
}

// a6 + a7, task = (slot, kDnRows output rows, pass of kDownPos positions);
// warp w owns rows 16 w .. 16 w + 15 of the block over the full K, so no
// partials are reduced. The pass's h is staged in shared memory as fp16
// (scaled into the fp16 range per position). The combine runs as its own
// kernel (every T this kernel serves).
template <int WFMT>
__global__ void __launch_bounds__(kRingThreads, kRingCtasPerSm) down_ring_kernel(ExpertArgs a, int stages, uint32_t stage_bytes) {
    griddep_wait();
    extern __shared__ __align__(128) uint8_t rsm[];
    RingHead* hd = reinterpret_cast<RingHead*>(rsm);
    float* hmul = reinterpret_cast<float*>(rsm + kRingHeadBytes);                       // [kDownPos]
    __half* hs = reinterpret_cast<__half*>(rsm + kRingHeadBytes + kDownPos * 4);        // [kDownPos][f]
    uint8_t* ring = rsm + kRingHeadBytes + kDownPos * 4 + dn_hs_bytes(a.f);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int KTf = a.f >> 7;
    const int units = a.d / kDnRows;
    const int hpitch = dn_hs_pitch(a.f);
    unsigned* ctr = a.ws.counters + kRingCtr + 2;
    constexpr int TSB = (WFMT == 0) ? 64 : 128;
    const uint32_t cb = 2u * kRingWarps * KTf * 512u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&hd->full[s], 1);
        mbar_fence_init();
    }
    ring_task_table(a, units, hd);
    const int ns = min(a.ws.meta[0], kRingMaxSlots);
    uint32_t fills = 0;
    bool out = false;
    int tnext = 0, tend = 0;   // kDnChunk consecutive tasks per grab
    auto issue = [&](int4 tk, int s) {
        dn_issue<WFMT>(a, tk, KTf, ring + s * stage_bytes, &hd->full[s]);
    };
    if (threadIdx.x == 0)
        for (; (int)fills < stages; ++fills)
            ring_fill(hd, stages, fills, ns, units, ctr, kDnChunk, tnext, tend, out, issue);
    int st_slot = -1, st_pass = -1;   // the (slot, pass) whose h is in hs
    for (int i = 0;; ++i) {
        if (!ring_acquire(hd->full, stages, i, a.ws.status)) break;
        const int4 tk = hd->task[i % stages];
        if (tk.x < 0) break;
        const int slot = tk.x, blk = tk.y, n0 = tk.z * kDownPos;
        const int e = a.ws.slot_expert[slot];
        const int p0 = a.ws.slot_off[slot], cnt = a.ws.slot_cnt[slot];
        const bool shared = (e == a.E);
        const float tsd = a.tscale[e * 3 + 2];
        const uint8_t* st = ring + (i % stages) * stage_bytes;
        const uint8_t* sc_ = st;          // codes of the block's tile rows
        const uint8_t* ss_ = st + cb;     // their scales
        const int np = min(kDownPos, cnt - n0);
        const int nb = (np + 7) >> 3;
        if (slot != st_slot || tk.z != st_pass) {
            // stage the pass's h once for the consecutive row blocks of one
            // (slot, pass) this CTA takes: 8 float4 loads in flight per thread
            if (threadIdx.x < np)
                hmul[threadIdx.x] = f16_range_mult(__uint_as_float(a.ws.hamax[p0 + n0 + threadIdx.x]));
            __syncthreads();
            const int row_f4 = a.f >> 2, total = np * row_f4;
            const float4* src = reinterpret_cast<const float4*>(a.ws.hf + (size_t)(p0 + n0) * a.f);
            for (int q0 = threadIdx.x; q0 < total; q0 += 8 * kRingThreads) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int q = q0 + u * kRingThreads;
                    if (q < total) v[u] = __ldcg(src + q);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int q = q0 + u * kRingThreads;
                    if (q < total) {
                        const float m = hmul[q / row_f4];
                        *reinterpret_cast<uint2*>(hs + (size_t)(q / row_f4) * hpitch + (q % row_f4) * 4) =
                            make_uint2(pack_half2(v[u].x * m, v[u].y * m), pack_half2(v[u].z * m, v[u].w * m));
                    }
                }
            }
            __syncthreads();
            st_slot = slot;
            st_pass = tk.z;
        }
        float acc[kNB][4];
#pragma unroll
        for (int q = 0; q < kNB; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[q][j] = 0.f;
        for (int kt = 0; kt < KTf; ++kt) {
            const uint4 wg = *reinterpret_cast<const uint4*>(sc_ + ((2 * warp) * KTf + kt) * 512 + lane * 16);
            const uint4 wh = *reinterpret_cast<const uint4*>(sc_ + ((2 * warp + 1) * KTf + kt) * 512 + lane * 16);
            const TileScales<WFMT> sc = lds_scales<WFMT>(ss_ + ((2 * warp) * KTf + kt) * TSB,
                                                         ss_ + ((2 * warp + 1) * KTf + kt) * TSB, g);
            uint32_t fa[8][4];
            decode_tile<WFMT>(wg, wh, sc, fa);
#pragma unroll
            for (int nt = 0; nt < kNB; ++nt) {
                if (nt >= nb) break;
                const int pl = nt * 8 + g;
                uint32_t b[16];
                if (pl < np) {
                    const uint4* hp = reinterpret_cast<const uint4*>(hs + (size_t)pl * hpitch + kt * 128 + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 v = hp[q];
                        b[4 * q + 0] = v.x;
                        b[4 * q + 1] = v.y;
                        b[4 * q + 2] = v.z;
                        b[4 * q + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) b[q] = 0u;
                }
                float sx[4][2];
                if constexpr (WFMT == 1) block_sums_q41(b, sx);
                mma_k128<WFMT>(acc[nt], fa, b, sc, sx);
            }
        }
        __syncthreads();   // every thread is done with the stage's weights and with hs
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            ring_fill(hd, stages, fills, ns, units, ctr, kDnChunk, tnext, tend, out, issue);
            ++fills;
        }
        // rows g, g + 8 of this warp's 16; positions 2c, 2c + 1 of each n-tile
#pragma unroll
        for (int nt = 0; nt < kNB; ++nt) {
            if (nt >= nb) break;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int n = n0 + nt * 8 + 2 * c + q;
                if (n >= cnt) continue;
                const int pos = p0 + n;
                const float wr = shared ? 1.0f : a.ws.w[__ldg(a.ws.perm + pos)];
                const float sc2 = tsd / hmul[n - n0] * wr;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int row = blk * kDnRows + warp * 16 + g + hh * 8;
                    a.ws.yw[(size_t)pos * a.d + row] = acc[nt][hh * 2 + q] * sc2;
                }
            }
        }
        __syncthreads();   // hmul read
    }
    if (threadIdx.x == 0) ring_exit(hd, stages, fills, ctr, a.ws.status);
}

__global__ void __launch_bounds__(256) combine_kernel(ExpertArgs a) {
    griddep_wait();
    const int rows_per_cta = 256;
    const int nblk = (a.d + rows_per_cta - 1) / rows_per_cta;
    const int t = blockIdx.x / nblk;
    const int row0 = (blockIdx.x % nblk) * rows_per_cta;
    const int row = row0 + threadIdx.x;
    if (t >= a.T || row >= a.d) return;
    float v = 0.f;
    if (a.n_shared) v = a.ws.yw[(size_t)(a.T * a.k + t) * a.d + row];
    for (int j = 0; j < a.k; ++j) {
        const int pos = a.ws.inv[t * a.k + j];
        v += a.ws.yw[(size_t)pos * a.d + row];
    }
    __nv_bfloat16 o = __float2bfloat16_rn(v);
    if (a.residual != nullptr) {
        const float r = __bfloat162float(a.residual[(size_t)t * a.d + row]);
        o = __float2bfloat16_rn(r + __bfloat162float(o));
    }
    a.out[(size_t)t * a.d + row] = o;
}

}  // namespace

namespace {

ExpertArgs make_args(const Shape& s, const LayerDev& L, int T, const Workspace& ws) {
    ExpertArgs a;
    a.codes = L.codes;
    a.scales = L.scales;
    a.tscale = L.tscale;
    a.codes_per_mat = s.codes_per_matrix();
    a.scales_per_mat = s.scales_per_matrix();
    a.d = s.d;
    a.f = s.f;
    a.E = s.E;
    a.k = s.k;
    a.n_shared = s.n_shared;
    a.T = T;
    a.ws = ws;
    a.out = nullptr;
    a.residual = nullptr;
    a.fuse_combine = (T <= kFuseCombineT) ? 1 : 0;
    return a;
}

int grid_for(int tasks) {
    const int cap = 148 * 8;
    return tasks < cap ? tasks : cap;
}

}  // namespace

namespace {

// The ring kernels serve kFuseCombineT < T <= kSmallT wherever their stages
// fit shared memory (at smaller T the register-streaming kernels, which fuse
// the combine, measured faster); FLINT_MOE_RING_EXPERTS=0 keeps the
// register-streaming kernels there too.
bool ring_enabled() {
    const char* env = getenv("FLINT_MOE_RING_EXPERTS");
    return !(env != nullptr && env[0] == '0');
}

int ring_grid(int max_tasks, int n_sms) { return max_tasks < n_sms ? max_tasks : n_sms; }

}  // namespace

int expert_launches(const Shape& s, int T) {
    const bool ring = T > kFuseCombineT && T <= kSmallT && dn_layout(s).stages >= 2 && ring_enabled();
    return 1 + ((T <= kFuseCombineT && !ring) ? 1 : 2);
}

cudaError_t prepare_experts() {
    const void* fns[4] = {(const void*)gateup_ring_kernel<0>, (const void*)gateup_ring_kernel<1>,
                          (const void*)down_ring_kernel<0>, (const void*)down_ring_kernel<1>};
    for (const void* fn : fns) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingSmemCap);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Every kernel of the decode-path chain (router, gate/up, down, combine) is
// launched with programmatic serialisation and waits for its predecessor at
// its first statement (pdl.cuh).
cudaError_t launch_gateup(const Shape& s, const LayerDev& L, int T, const Workspace& ws,
                          cudaStream_t st, int* n_launch) {
    ExpertArgs a = make_args(s, L, T, ws);
    const int max_slots = min(s.E, T * s.k) + s.n_shared;
    const RingLayout rl = gu_layout(s);
    *n_launch += 1;
    if (T > kFuseCombineT && T <= kSmallT && rl.stages >= 2 && ring_enabled()) {
        int dev = 0, n_sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        const int grid = ring_grid(max_slots * (s.f / 16), kRingCtasPerSm * n_sms);
        if (s.wfmt == 0)
            return launch_pdl(gateup_ring_kernel<0>, dim3(grid), dim3(kRingThreads), rl.smem, st, a, rl.stages,
                              rl.stage_bytes);
        return launch_pdl(gateup_ring_kernel<1>, dim3(grid), dim3(kRingThreads), rl.smem, st, a, rl.stages,
                          rl.stage_bytes);
    }
    const int max_pass = (T + 8 * kNB - 1) / (8 * kNB);
    const int grid = grid_for(max_slots * (s.f / 16) * max_pass);
    if (s.wfmt == 0) return launch_pdl(gateup_kernel<0>, dim3(grid), dim3(kThreads), 0, st, a);
    return launch_pdl(gateup_kernel<1>, dim3(grid), dim3(kThreads), 0, st, a);
}

cudaError_t launch_down(const Shape& s, const LayerDev& L, int T, const Workspace& ws,
                        __nv_bfloat16* out, const __nv_bfloat16* residual, cudaStream_t st,
                        int* n_launch) {
    ExpertArgs a = make_args(s, L, T, ws);
    a.out = out;
    a.residual = residual;
    const int max_slots = min(s.E, T * s.k) + s.n_shared;
    const RingLayout rl = dn_layout(s);
    const bool ring = T > kFuseCombineT && T <= kSmallT && rl.stages >= 2 && ring_enabled();
    cudaError_t e;
    if (ring) {
        a.fuse_combine = 0;   // the ring kernel leaves the combine to its own kernel
        int dev = 0, n_sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        const int grid = ring_grid(max_slots * (s.d / kDnRows), kRingCtasPerSm * n_sms);
        if (s.wfmt == 0)
            e = launch_pdl(down_ring_kernel<0>, dim3(grid), dim3(kRingThreads), rl.smem, st, a, rl.stages,
                           rl.stage_bytes);
        else
            e = launch_pdl(down_ring_kernel<1>, dim3(grid), dim3(kRingThreads), rl.smem, st, a, rl.stages,
                           rl.stage_bytes);
    } else {
        const int max_pass = (T + kDownPos - 1) / kDownPos;
        const int grid = grid_for(max_slots * (s.d / 64) * max_pass);
        if (s.wfmt == 0)
            e = launch_pdl(down_kernel<0>, dim3(grid), dim3(kThreads), 0, st, a);
        else
            e = launch_pdl(down_kernel<1>, dim3(grid), dim3(kThreads), 0, st, a);
    }
    *n_launch += 1;
    if (e == cudaSuccess && !a.fuse_combine) {
        const int nblk = (s.d + 255) / 256;
        e = launch_pdl(combine_kernel, dim3(T * nblk), dim3(256), 0, st, a);
        *n_launch += 1;
    }
    return e;
}

}  // namespace flint
