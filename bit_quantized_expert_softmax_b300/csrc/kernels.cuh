// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace flint {

// Device-resident weights of one layer, in the kernels' tiled layout.
//
// Codes of a matrix [R x K] are stored as tiles of 8 rows x 128 K, tile
// (rt, kt) at byte offset (rt*(K/128) + kt)*512. Inside a tile, lane
// l = 4g + c owns 16 bytes at offset l*16; byte 2s (s = 0..7) is canonical
// byte kt*64 + 8s + c of row rt*8 + g (K elements 16s+2c, 16s+2c+1 of the
// tile) and byte 2s+1 is canonical byte kt*64 + 8s + c + 4 (K elements
// 16s+2c+8, 16s+2c+9). This is the A-fragment order of mma.m16n8k16, so one
// 16-byte load per lane and tile feeds 8 mma steps.
//
// NVFP4 block scales: per tile 64 bytes, [g][s] = scale of row rt*8+g for the
// 16 K elements of step s. q4_1: per tile 128 bytes, [g][b] = 4 bytes
// (fp16 d, fp16 m) of row rt*8+g for K block kt*4+b (32 elements).
struct LayerDev {
    float* router = nullptr;        // [E][d]
    float* bias = nullptr;          // [E] (zeros when absent)
    uint8_t* codes = nullptr;       // [n_slots][3][f*d/2] tiled
    uint8_t* scales = nullptr;      // [n_slots][3][scale bytes] tiled
    float* tscale = nullptr;        // [n_slots][3]
    __nv_bfloat16* router_hi = nullptr;   // [E][d] bf16(W_r)
    __nv_bfloat16* router_lo = nullptr;   // [E][d] bf16(W_r - bf16(W_r))
    CUtensorMap tmap_router_hi, tmap_router_lo;   // 128x64 swizzled boxes of the two
    bool umma_router = false;
    uint8_t* prefill = nullptr;     // swizzled FP4 tiles of all experts (large-T path), or null
    float* router_t = nullptr;      // [d][E] W_r transposed (the one-launch decode stack), or null
    bool loaded = false;
};

// One layer of the one-launch decode stack (a device table of these, in
// stack order).
struct StackLayer {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* tscale;
    const float* router_t;   // [d][E]
    const float* bias;       // [E]
};

struct Shape {
    int d, f, E, k, n_shared, wfmt, max_tokens;
    int n_slots() const { return E + n_shared; }
    size_t codes_per_matrix() const { return (size_t)f * d / 2; }
    size_t scales_per_matrix() const {
        return wfmt == 0 ? (size_t)f * d / 16 : (size_t)f * d / 32 * 4;
    }
    int positions(int T) const { return T * (k + n_shared); }
};

// Device bytes of a layer's tensor-scale array ([n_slots][3] fp32), padded to
// 256 bytes so that it can be bulk-copied whole.
inline size_t tscale_bytes(const Shape& s) { return ((size_t)s.n_slots() * 12 + 255) / 256 * 256; }

// Per-handle scratch for one forward (sized for max_tokens).
struct Workspace {
    float* logits;        // [Tm][E]
    int* idx;             // [Tm][k]
    float* w;             // [Tm][k]
    int* perm;            // [Tm*k]  sorted position -> assignment t*k+j
    int* inv;             // [Tm*k]  assignment -> sorted position
    int* offsets;         // [E+1]
    int* ecount;          // [E * kEcountStride] per-expert assignment counters of the FP4 path, one per
                          //        128-byte line (zero between forwards)
    int* slot_expert;     // [E+1]  active slot -> expert (E = shared)
    int* slot_off;        // [E+1]  first position of the slot
    int* slot_cnt;        // [E+1]  positions of the slot
    int* meta;            // [8]    0: number of active slots
    __half* x16;          // [Tm][d]  fp16 hidden, scaled per token, fragment-permuted
    float* xinv;          // [Tm]     inverse of the per-token fp16 scale
    float* hf;            // [P][f]   expert intermediate h (fp32, fragment-permuted)
    uint32_t* hamax;      // [P]      max |h| per position (float bits)
    float* yw;            // [P][d]   weighted expert outputs
    int* chunk_hist;      // [n_chunks][E]
    uint32_t* counters;   // [kCounters] arrival counters (self-resetting)
    uint32_t* gbar;       // [64]  grid-barrier count ([0]) and generation ([32])
    uint32_t* dbg;        // [64]  the timeout check's own barrier counter
    unsigned long long* gbar8;  // [kGridGroups * kGridGroupStride] the decode stack's grid-barrier counters
    unsigned long long* racc;   // [2][kRaccCopies][kFusedMaxT][E] fixed-point router logits of the decode stack
    uint32_t* rnf;              // [2][kRaccCopies][kFusedMaxT][E] their non-finite flags
    uint32_t* status;     // device status word
};

// Global scratch of the single-launch decode kernel.
struct FusedScratch {
    float* logits;        // [T][E]
    float* h;             // [T][k+1][f]
    uint32_t* bar;        // [64], zero-initialised
    uint32_t* status;
};

constexpr int kCounters = 1024;
constexpr int kBucketChunk = 2048;      // assignments per bucketing CTA
constexpr int kEcountStride = 32;       // ints between two experts' counters in ws.ecount
constexpr int kRaccCopies = 8;          // copies of the decode stack's router accumulators (atomics spread)
constexpr int kSmallT = 64;             // fused router (logits + top-k + bucketing) up to this many tokens
constexpr int kFuseCombineT = 8;        // combine in the down kernel's last CTA up to this many tokens

// router.cu
cudaError_t prepare_router();   // once per device: shared-memory opt-in of the fused router
bool router_fused(const Shape& s, int T);   // router, top-k and bucketing in one launch
int expert_launches(const Shape& s, int T);   // gate/up + down (+ combine) kernels of the mma.sync path
cudaError_t prepare_experts();  // once per device: shared-memory opt-in of the ring-fed expert kernels
cudaError_t launch_router(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                          const Workspace& ws, cudaStream_t st, int* n_launch, bool stage_x16 = true);
cudaError_t launch_topk(const float* logits, int T, int E, int k, int* idx, float* w,
                        cudaStream_t st);
// the FP4 path's routing: logits, top-k and per-expert ranks (ws.inv, ws.ecount)
cudaError_t launch_router_fp4(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T, const Workspace& ws,
                              cudaStream_t st, int* n_launch);
cudaError_t launch_bucket(const Shape& s, const int* idx, int T, const Workspace& ws,
                          cudaStream_t st, int* n_launch, bool reset_hamax = true);

// experts.cu: gate/up (one launch), then down + combine (one or two launches)
cudaError_t launch_gateup(const Shape& s, const LayerDev& L, int T, const Workspace& ws,
                          cudaStream_t st, int* n_launch);
cudaError_t launch_down(const Shape& s, const LayerDev& L, int T, const Workspace& ws,
                        __nv_bfloat16* out, const __nv_bfloat16* residual, cudaStream_t st,
                        int* n_launch);

// decode_fused.cu: one persistent launch per layer for T <= kFusedMaxT
constexpr int kFusedMaxT = 2;
size_t fused_smem_bytes(const Shape& s, int T, int n_sms, int* n_slots_out, int offs[10]);
cudaError_t prepare_decode_fused();   // once per device: shared-memory opt-in
// the whole decode stack in one cooperative launch (T <= kFusedMaxT); 0 if
// its shared-memory plan does not fit
size_t stack_smem_bytes(const Shape& s, int T, int n_sms);
cudaError_t launch_decode_stack(const Shape& s, const StackLayer* layers_dev, int n_layers, __nv_bfloat16* x, int T,
                                const FusedScratch& fs, unsigned long long* gbar8, unsigned long long* racc,
                                uint32_t* rnf, int n_sms, cudaStream_t st);
cudaError_t transpose_router(const float* w, float* wt, int E, int d, cudaStream_t st);
cudaError_t launch_decode_fused(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                                __nv_bfloat16* out, const __nv_bfloat16* residual, const FusedScratch& fs,
                                int n_sms, cudaStream_t st, const LayerDev* next = nullptr);

// prefill_fp4.cu: tensor-core kernels for large T
cudaError_t prepare_prefill();   // once per device: shared-memory opt-in
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rows, int cols);
bool router_umma_supported(const Shape& s);
cudaError_t split_router(const float* w, __nv_bfloat16* hi, __nv_bfloat16* lo, size_t n, cudaStream_t st);
cudaError_t launch_router_umma(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T, float* logits,
                               uint32_t* status, cudaStream_t st);

// moe_prefill.cu: block-scaled FP4 expert projections for large T
bool prefill_fp4_supported(const Shape& s);
size_t prefill_weight_bytes(const Shape& s);
size_t prefill_workspace_bytes(const Shape& s, int Tm);
cudaError_t prepare_prefill_fp4();
cudaError_t pack_prefill_weights(const Shape& s, const uint8_t* codes, const uint8_t* scales, uint8_t* dst,
                                 cudaStream_t st);
cudaError_t launch_prefill_experts(const Shape& s, const LayerDev& L, const __nv_bfloat16* x, int T,
                                   const Workspace& ws, uint8_t* pw, int Tm, __nv_bfloat16* out,
                                   const __nv_bfloat16* residual, cudaStream_t st, int* n_launch,
                                   const cudaEvent_t* marks);
cudaError_t launch_act_quant(const __nv_bfloat16* x, int T, int K, uint8_t* codes, uint8_t* scales, float* rowscale,
                             cudaStream_t st);

// gemm_fp4.cu: swizzled-tile packing for the block-scaled FP4 GEMM
cudaError_t pack_fp4_tiles(const uint8_t* codes, const uint8_t* scales, uint8_t* blocks, int R, int K,
                           cudaStream_t st);
cudaError_t prepare_gemm_fp4();

// lm_head.cu: the 4-bit output head and its sampling front-end
constexpr int kHeadMaxT = 8;      // tokens per head call (the MMA's 8 token columns)
constexpr int kHeadMaxD = 4096;   // hidden width the head's shared-memory plan covers
struct HeadScratch {
    uint32_t* cand_key;       // [kHeadMaxT][parts][32] candidates of the sampler's parts
    uint32_t* cand_idx;
    unsigned int* counters;   // [kHeadMaxT], zero between calls
};
size_t head_smem_bytes(int T, int d);
cudaError_t prepare_head();
cudaError_t launch_head_gemv(const uint8_t* codes, const uint8_t* scales, float tscale, const __nv_bfloat16* x,
                             int T, int d, int V, float* logits, int n_sms, cudaStream_t st);
int head_sample_parts(int V);
bool head_sample_supported(int V, int top_k);
cudaError_t launch_head_sample(const float* logits, int T, int V, float temperature, int top_k, float top_p,
                               const float* u, int* tokens, int* topk_idx, const HeadScratch& hs, uint32_t* status,
                               cudaStream_t st);

// debug_wait.cu: bounded waits that run out (kind 0 mbarrier, 1 grid barrier)
cudaError_t launch_wait_timeout(int kind, uint32_t limit, unsigned long long* count, uint32_t* status,
                                cudaStream_t st);

// fp4_peak.cu: dense block-scaled FP4 tensor-core throughput probe
cudaError_t launch_fp4_peak(int n, int iters, int n_sms, uint32_t* status, cudaStream_t st);

// repack.cu
cudaError_t launch_repack_matrix(const uint8_t* codes_src, const uint8_t* scales_src,
                                 uint8_t* codes_dst, uint8_t* scales_dst, int R, int K, int wfmt,
                                 cudaStream_t st);
cudaError_t launch_dequant_matrix(const uint8_t* codes, const uint8_t* scales, float tscale_host,
                                  const float* tscale_dev, int R, int K, int wfmt, float* out,
                                  cudaStream_t st);

}  // namespace flint
