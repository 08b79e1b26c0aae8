/*
 * flint_moe.h -- C ABI of the B300 (sm_103a) sparse 4-bit MoE FFN layer.
 *
 * The layer is the conditional FFN of a Flint-shaped model ("Recursive Flint
 * 40B-A2.5B: a coding model designed speed-first", orcarouter.ai blog,
 * section "The architecture is an argument about memory bandwidth", Sparsity
 * bullet): per MoE layer 256 routed experts with 6 chosen per token plus one
 * always-on shared expert; 47 of the model's 49 layers are MoE layers. The
 * experts carry 4-bit weights, NVFP4 or q4_1 (section "What actually
 * shipped"). For one layer and tokens x[t] (bfloat16, width d):
 *
 *   L[t,e]  = sum_i x[t,i] W_r[e,i] + b[e]                  fp32 router logits
 *   S_t     = 6 largest logits (ties: lower expert index), descending
 *   w[t,j]  = softmax(L[t,:])[S_t[j]] / sum_{e in S_t} softmax(L[t,:])[e]
 *   y_e(x)  = W_down_e ( silu(W_gate_e x) * (W_up_e x) ),  silu(z) = z/(1+e^-z)
 *   out[t]  = bf16( y_shared(x[t]) + sum_j w[t,j] y_{S_t[j]}(x[t]) )
 *
 * Weight formats (canonical host layout accepted by flint_moe_load_weights):
 *   NVFP4: w = E2M1(code) * E4M3(block scale) * fp32 tensor scale; one E4M3
 *          block scale per 16 consecutive elements of a row, one fp32 tensor
 *          scale per matrix. Two codes per byte, element 2i in the low nibble.
 *   q4_1 : w = d*q + m, q in 0..15; per 32 consecutive elements of a row one
 *          fp16 d followed by one fp16 m (little endian, 4 bytes). Codes as
 *          for NVFP4.
 * Matrices per expert: 0 = gate [f x d], 1 = up [f x d], 2 = down [d x f],
 * each row-major with the contraction axis (K) contiguous.
 *
 * Conventions shared by every call:
 *   - Pointers named *_dev are CUDA device pointers on the handle's device;
 *     all others are host pointers. The caller owns every buffer it passes.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls that
 *     take a stream only enqueue work and return; results are ready once the
 *     stream reaches that point.
 *   - Errors are returned, never thrown. FLINT_EINVAL / FLINT_ESTATE mean
 *     nothing was enqueued. Faults detected on the device (non-finite router
 *     logits, out-of-range indices) set a status word that flint_moe_status
 *     reports and clears.
 *   - A handle is not safe for concurrent use from several host threads, and
 *     two forwards on one handle must not overlap on the GPU (they share one
 *     workspace).
 */
#ifndef FLINT_MOE_H
#define FLINT_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FLINT_API __attribute__((visibility("default")))
#else
#define FLINT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct flint_moe flint_moe;

typedef enum {
    FLINT_OK = 0,
    FLINT_EINVAL = 1,    /* bad argument: NULL, size, alignment, range */
    FLINT_ENOMEM = 2,    /* device allocation failed */
    FLINT_ECUDA = 3,     /* a CUDA runtime call or launch failed */
    FLINT_ESTATE = 4,    /* handle not ready (weights of the layer not loaded) */
    FLINT_ETIMEOUT = 5,  /* a bounded device-side wait gave up */
    FLINT_ENOTIMPL = 6,  /* configuration not supported by this build */
    FLINT_EDEVICE = 7    /* the device reported a data fault (see flint_moe_status) */
} flint_status;

typedef enum { FLINT_W_NVFP4 = 0, FLINT_W_Q4_1 = 1 } flint_wfmt;

/* Shape of the layers held by one handle. Constraints: d and f multiples of
 * 128; 32 <= n_experts <= 256 and a multiple of 32; 1 <= top_k <= 8 and
 * top_k <= n_experts; n_shared 0 or 1; 1 <= max_tokens <= 65536;
 * n_layers >= 1. The Flint shape is d=2048, f=512, n_experts=256, top_k=6,
 * n_shared=1, n_layers=47. */
typedef struct {
    int d;
    int f;
    int n_experts;
    int top_k;
    int n_shared;
    int wfmt;        /* flint_wfmt */
    int max_tokens;  /* largest T any forward on this handle will pass */
    int n_layers;
    int device;      /* CUDA device ordinal */
} flint_moe_config;

/* One layer's weights, canonical host layout (see the format notes above).
 * n = n_experts + n_shared expert slots; the shared expert is slot n_experts.
 *   router        float  [n_experts][d]          one row per expert
 *   router_bias   float  [n_experts] or NULL (all zero)
 *   codes         uint8  [n][3][f*d/2]
 *   scales        uint8  [n][3][f*d/16]   (NVFP4: E4M3 bytes)
 *                        [n][3][f*d/32*4] (q4_1: fp16 d, fp16 m per block)
 *   tensor_scale  float  [n][3] (NVFP4); ignored for q4_1 (may be NULL)
 * E4M3 block scales must be non-negative and not NaN (bytes 0x00..0x7E); fp16
 * d and m, the router, its bias and the tensor scales must be finite. */
typedef struct {
    const float* router;
    const float* router_bias;
    const uint8_t* codes;
    const uint8_t* scales;
    const float* tensor_scale;
} flint_moe_weights;

/* Create a handle on cfg->device: validates cfg and allocates the per-token
 * workspace for cfg->max_tokens (no weights yet). *out is NULL on failure.
 * Errors: FLINT_EINVAL (cfg), FLINT_ENOTIMPL, FLINT_ENOMEM, FLINT_ECUDA. */
FLINT_API flint_status flint_moe_create(const flint_moe_config* cfg, flint_moe** out);

/* Copy layer `layer`'s weights from host memory into device memory owned by
 * the handle and repack them into the kernels' tiled layout. Synchronous: the
 * host buffers may be freed on return. Loading a layer again replaces it.
 * Errors: FLINT_EINVAL (NULL pointer, layer out of range, NaN/negative E4M3
 * scale, non-finite fp16 or fp32 value), FLINT_ENOMEM, FLINT_ECUDA. */
FLINT_API flint_status flint_moe_load_weights(flint_moe* h, int layer, const flint_moe_weights* w);

/* One MoE layer: out_dev[T][d] = MoE_layer(hidden_dev[T][d]), both bfloat16,
 * 16-byte aligned, not overlapping. T == 0 is a no-op returning FLINT_OK.
 * The kernels are enqueued on `stream` (a cudaStream_t; NULL: the legacy
 * default stream) and keep its order: work enqueued before the call completes
 * before any kernel of the layer reads or writes memory, and work enqueued
 * after it sees the output. (The multi-kernel paths launch their kernels with
 * programmatic stream serialisation: a kernel may be scheduled while the one
 * before it is finishing, but waits for it before touching memory.)
 * Errors: FLINT_EINVAL (NULL, misaligned, T < 0 or T > max_tokens, layer out
 * of range), FLINT_ESTATE (layer not loaded), FLINT_ECUDA (launch). */
FLINT_API flint_status flint_moe_forward(flint_moe* h, int layer, const void* hidden_dev, int T,
                               void* out_dev, void* stream);

/* Decode stack with residual: for l = layer0 .. layer0+n_layers-1,
 *   x <- bf16( x + MoE_layer_l(x) )   (the sum taken in fp32 of the bf16 values)
 * applied in place to hidden_dev[T][d] (bfloat16, 16-byte aligned). Same
 * errors as flint_moe_forward. For T <= 2 (with one shared expert) all
 * n_layers layers run as ONE kernel launch: a persistent cooperative kernel
 * with two grid barriers per layer, which computes each layer's router logits
 * from the previous layer's output rows as they are produced (summed in 64-bit
 * fixed point, 2^-32 units, so the result does not depend on arrival order).
 * Setting FLINT_MOE_STACK_KERNEL=0 before flint_moe_create runs each layer as
 * one forward instead (the single-launch decode kernel, one launch per layer;
 * the same result as chaining flint_moe_forward bit for bit); other T always
 * run that way.
 * Enqueues only kernels, so the whole call can be captured into a CUDA graph. */
FLINT_API flint_status flint_moe_forward_stack(flint_moe* h, int layer0, int n_layers, void* hidden_dev,
                                     int T, void* stream);

/* Release the handle and all device memory it owns. NULL-safe. Synchronises
 * the device first. */
FLINT_API void flint_moe_destroy(flint_moe* h);

/* Wait for the device, then read and clear the handle's device status word.
 * FLINT_OK if no fault was recorded; FLINT_EDEVICE if a kernel recorded a
 * data fault (non-finite router logit); FLINT_ETIMEOUT if a bounded wait gave
 * up; FLINT_ECUDA if the device reports a CUDA error. */
FLINT_API flint_status flint_moe_status(flint_moe* h);

/* Static description of a status code. */
FLINT_API const char* flint_moe_status_string(flint_status s);

/* ---- per-step entry points (the same kernels the forward runs) ---------- */

/* Router of one layer (steps a1-a2): logits_dev[T][n_experts] fp32,
 * idx_dev[T][top_k] int32 (descending logit, ties to the lower index),
 * w_dev[T][top_k] fp32 renormalised softmax weights. Any output pointer may
 * be NULL. Errors as flint_moe_forward. */
FLINT_API flint_status flint_moe_router(flint_moe* h, int layer, const void* hidden_dev, int T,
                              float* logits_dev, int32_t* idx_dev, float* w_dev, void* stream);

/* Top-k selection and renormalised softmax weights on given fp32 logits
 * (step a2). logits_dev [T][E]; idx_dev [T][k]; w_dev [T][k] (may be NULL).
 * Needs no handle. Constraints: E multiple of 32 in 32..256, 1 <= k <= 8,
 * T >= 0. Non-finite logits rank below every finite one; they are not
 * reported here. */
FLINT_API flint_status flint_moe_topk(const float* logits_dev, int T, int E, int k, int32_t* idx_dev,
                            float* w_dev, void* stream);

/* Token -> expert bucketing (step a3) of idx_dev[T][k] (values in 0..E-1):
 * offsets_dev[E+1] exclusive prefix sum of the per-expert counts,
 * perm_dev[T*k] the flat assignments a = t*k + j ordered by (expert, a).
 * Uses the handle's workspace (T <= max_tokens, k == top_k, E == n_experts).
 * Out-of-range expert indices set the device status word (FLINT_EDEVICE) and
 * are dropped. */
FLINT_API flint_status flint_moe_bucket(flint_moe* h, const int32_t* idx_dev, int T, int32_t* offsets_dev,
                              int32_t* perm_dev, void* stream);

/* Dequantise one matrix of one expert of a loaded layer from the device
 * layout back to fp32 in canonical order: out_dev[R][K] with [R, K] =
 * [f, d] (mat 0 gate, 1 up) or [d, f] (mat 2 down); expert == n_experts is the
 * shared expert. NVFP4 values are fp32(E2M1 * E4M3 * tensor scale), q4_1
 * values fp32(d*q + m), each rounded once, computed with the decoders the
 * expert kernels use. The kernels never round a weight: they multiply by the
 * exact E2M1 * E4M3 product (fp16) and apply the tensor scale to the fp32
 * accumulator; for q4_1 they multiply by the exact codes q and add
 * d * sum(q x) + m * sum(x) per 32-element block, the regrouped d*q + m.
 * Errors as flint_moe_forward. */
FLINT_API flint_status flint_moe_dequant(flint_moe* h, int layer, int expert, int mat, float* out_dev,
                               void* stream);

/* Bytes of device memory the handle holds (weights + workspace). */
FLINT_API size_t flint_moe_device_bytes(const flint_moe* h);

/* Which 5th-generation tensor-core (tcgen05) kernels a single-layer forward
 * of T tokens on this loaded layer uses: bit 0 = router logits GEMM, bit 1 =
 * block-scaled FP4 expert GEMMs. 0 when neither; -1 on bad arguments.
 * Bit 1 is set for T > 64 on NVFP4 weights with d = 2048, f = 512 and one
 * shared expert when max_tokens > 64; that path quantises the activations
 * entering each expert projection to NVFP4 (flint_moe_debug_act_quant; h is
 * quantised from its fp32 value), so its result is the W4A4 product, not the W4A16
 * one the other paths compute. Setting FLINT_MOE_TCGEN05_PREFILL=0 before
 * flint_moe_create turns all these kernels off for the handle (the mma.sync
 * and CUDA-core paths remain); FLINT_MOE_FP4_EXPERTS=0 turns off only the
 * FP4 expert GEMMs. */
FLINT_API int flint_moe_tensor_core_plan(const flint_moe* h, int layer, int T);

/* Block-scaled FP4 matrix product on the 5th-generation tensor cores, through
 * the same kernel the large-T expert projections use: d_dev[M][N] (fp32) =
 * A . B^T with A [M][K] and B [N][K] in canonical NVFP4 layout (codes
 * [rows][K/2], element 2i in the low nibble; E4M3 scales [rows][K/16]; no
 * tensor scale), all device pointers, 16-byte aligned. M and N multiples of
 * 128, K a multiple of 256. Synchronous; allocates and frees temporary device
 * memory for the packed tiles. Errors: FLINT_EINVAL (sizes, NULL),
 * FLINT_ENOMEM, FLINT_ECUDA, FLINT_ETIMEOUT (a bounded device wait gave up). */
FLINT_API flint_status flint_moe_debug_fp4_gemm(const uint8_t* a_codes_dev, const uint8_t* a_scales_dev,
                                                const uint8_t* b_codes_dev, const uint8_t* b_scales_dev, int M,
                                                int N, int K, float* d_dev, void* stream);

/* NVFP4 quantisation of bf16 activations exactly as the large-T expert path
 * applies it before its block-scaled FP4 GEMMs (T > 64, NVFP4 weights):
 * per row an fp32 scale s = amax/2688 (rowscale_dev[T]); per 16 elements an
 * E4M3 scale byte sb = E4M3_rne((amax_16/6)/s) (scales_dev[T][K/16]); codes
 * E2M1_rne(v * (1/(E4M3(sb)*s))) in fp32 (codes_dev[T][K/2], element 2i in
 * the low nibble). A zero row gives s = 0, zero scales and zero codes. The
 * pages fix only the weights' NVFP4 format ("Flint", the repository list of
 * the NVFP4 GGUF build); using it for the activations, with one fp32 scale per
 * token, is this library's reading, forced by the FP4 x FP4 tensor-core MMA
 * that NVFP4 weights take. K must be 2048 or 512; x_dev and codes_dev
 * 16-byte aligned, scales_dev 4-byte aligned. Asynchronous on `stream`.
 * Errors: FLINT_EINVAL (K, T < 0, NULL, misaligned), FLINT_ECUDA. */
FLINT_API flint_status flint_moe_debug_act_quant(const void* x_dev, int T, int K, uint8_t* codes_dev,
                                                 uint8_t* scales_dev, float* rowscale_dev, void* stream);

/* NVFP4 quantisation of one bf16 weight matrix on the GPU, into the canonical
 * NVFP4 layout flint_moe_load_weights and flint_moe_load_lm_head accept. The
 * Flint blog ships NVFP4 weights ("Recursive Flint 40B-A2.5B", section "What
 * actually shipped", NVFP4 GGUF bullet) and gives no quantisation procedure;
 * this is the activation rule of flint_moe_debug_act_quant with one fp32
 * tensor scale for the whole matrix: s = amax(|w|)/2688; per 16 consecutive
 * elements of a row sb = E4M3_rne((amax_16/6)/s); codes
 * E2M1_rne(w * (1/(E4M3(sb)*s))), all in fp32, ties to even, saturating.
 * w_dev: bf16 [R][K] (device, 16-byte aligned); codes_dev: [R][K/2], element
 * 2i in the low nibble (8-byte aligned); scales_dev: [R][K/16] E4M3 bytes;
 * tensor_scale_dev: one fp32 (4-byte aligned; used as scratch until the last
 * of the three kernels writes s). An all-zero matrix gives s = 0, zero
 * scales and codes. Asynchronous on `stream`. Errors: FLINT_EINVAL (R < 1, K
 * not a positive multiple of 16, NULL, misaligned), FLINT_ECUDA. */
FLINT_API flint_status flint_moe_quantize_nvfp4(const void* w_dev, int R, int K, uint8_t* codes_dev,
                                                uint8_t* scales_dev, float* tensor_scale_dev, void* stream);

/* ---- decode attention ------------------------------------------------------
 * One decode step of a Flint-shaped attention layer ("Recursive Flint
 * 40B-A2.5B", section "The architecture is an argument about memory
 * bandwidth", Attention and Position-encoding bullets): 32 query heads and 4
 * key-value heads of dimension 128; 35 sliding-window layers with a 513-token
 * window (the current token and the 512 before it) and 14 full-attention
 * layers; rotary positions on the sliding-window layers only; per-head QK
 * RMSNorm and learned per-head attention sinks. The blog gives no formulas;
 * the readings: q_h <- rmsnorm(q_h) * q_norm_w and k <- rmsnorm(k) * k_norm_w
 * over the head dimension (eps); rotation of the pairs (i, i+64) by
 * pos * theta^(-i/64) when rope = 1; scores q.k / sqrt(128) over the window's
 * keys (query head h reads key head h / 8); the sink logit joins the softmax
 * denominator only. */
typedef struct {
    int n_heads;       /* query heads: 8 per key-value head (32 in Flint) */
    int n_kv;          /* key-value heads (4 in Flint), 1..64 */
    int head_dim;      /* 128 */
    int window;        /* positions attended, the current one included: 513 for sliding-window layers, 0 = all */
    int cap;           /* cache slots per sequence and key-value head; position p lives in slot p % cap;
                          cap >= window for sliding-window layers, cap > every position for full attention */
    int rope;          /* 1: rotary positions (sliding-window layers); 0: none */
    float rope_theta;  /* rotary base (10000 here; the blog does not give it) */
    float eps;         /* RMSNorm epsilon (1e-6) */
} flint_moe_attn_config;

/* For each of B sequences, attend its new token at position pos_dev[b] (int32,
 * >= 0): q_dev bf16 [B][n_heads][128], k_dev and v_dev bf16 [B][n_kv][128]
 * (the projections, before norm and rotation); k_cache_dev and v_cache_dev
 * bf16 [B][n_kv][cap][128] (16-byte aligned) hold the keys (normed, rotated)
 * and values of earlier positions; q_norm_w_dev and k_norm_w_dev fp32 [128];
 * sinks_dev fp32 [n_heads]; out_dev bf16 [B][n_heads][128]. Reads the cache
 * slots of positions pos-1 down to the window's start, then writes the new
 * key (normed, rotated) and value, bf16, to slot pos % cap. The current token
 * attends to its own key and value unrounded. Arithmetic: the scores and the
 * weighted sum of values run on the tensor cores with fp32 accumulation; the
 * cached keys and values enter as stored (bf16), the normed query and the
 * softmax probabilities as bf16 hi + lo pairs (about 16 significant bits);
 * the softmax itself is fp32. All pointers are device pointers; asynchronous
 * on `stream`. Errors: FLINT_EINVAL (configuration,
 * B < 0, NULL, misaligned cache), FLINT_ECUDA. */
FLINT_API flint_status flint_moe_attn_decode(const flint_moe_attn_config* cfg, int B, const void* q_dev, const void* k_dev,
                                         const void* v_dev, void* k_cache_dev, void* v_cache_dev,
                                         const int32_t* pos_dev, const float* q_norm_w_dev,
                                         const float* k_norm_w_dev, const float* sinks_dev, void* out_dev,
                                         void* stream);

/* ---- the 4-bit output head and its sampler ---------------------------------
 * The Flint blog ("Recursive Flint 40B-A2.5B", section "The quantisation
 * recipe is the most transferable part") ships the output layer (lm_head)
 * quantised to 4 bits because it is a large share of the bytes read per
 * token; its serving defaults are temperature 1.0, top-p 0.95, top-k 20
 * (section "The three scores, and the footnotes that come with them",
 * Sampling bullet). */

/* Copy the NVFP4 output head W [vocab x d] into the handle, repacked for the
 * GEMV. Host pointers, canonical layout: codes uint8 [vocab][d/2] (two E2M1
 * codes per byte, low nibble first), scales uint8 [vocab][d/16] (one E4M3
 * byte per 16 codes of a row), tensor_scale fp32. The caller keeps ownership
 * of the host arrays. vocab must be a positive multiple of 8. A second call
 * replaces the head. Synchronises the device. FLINT_EINVAL on bad arguments,
 * FLINT_ENOMEM / FLINT_ECUDA on device failures. */
FLINT_API flint_status flint_moe_load_lm_head(flint_moe* h, int vocab, const void* codes, const void* scales,
                                    float tensor_scale);

/* logits_dev[t][v] = sum_i x[t][i] * W[v][i] for T <= 8 tokens of
 * hidden_dev (bf16 [T][d], device, 16-byte aligned) into logits_dev (fp32
 * [T][vocab], device, 16-byte aligned). Weights decoded to fp16 exactly,
 * x rounded to fp16 after a power-of-two scale per token, fp32 accumulation.
 * Asynchronous on `stream`. FLINT_ESTATE if no head is loaded, FLINT_EINVAL
 * for T outside 0..8 or bad pointers (T = 0 does nothing). */
FLINT_API flint_status flint_moe_lm_head(flint_moe* h, const void* hidden_dev, int T, float* logits_dev,
                               void* stream);

/* Draw one token per row of logits_dev (fp32 [T][vocab], device; the loaded
 * head's vocab). temperature <= 0: the largest logit (equal logits: the lower
 * index). Otherwise: the top_k largest logits (descending, ties to the lower
 * index); softmax over them at the temperature; the smallest prefix whose
 * probability reaches top_p (a member is kept while the sum of the ones
 * before it is below top_p); the first kept member whose cumulative
 * probability exceeds u[t] times the kept total. u_dev: fp32 [T] uniforms in
 * [0, 1) (device), tokens_dev: int32 [T] (device); topk_dev, if not NULL,
 * receives the top_k indices per token (int32 [T][top_k]; only entry 0 when
 * temperature <= 0). 1 <= top_k <= 32, 0 < top_p <= 1, T <= 8, and
 * ceil(vocab / 2048) * top_k <= 2048. NaN logits rank last and set
 * FLINT_EDEVICE in the status word. Asynchronous on `stream`; calls on one
 * handle must not overlap on the GPU (they share the handle's scratch). */
FLINT_API flint_status flint_moe_sample(flint_moe* h, const float* logits_dev, int T, float temperature,
                              int top_k, float top_p, const float* u_dev, int32_t* tokens_dev,
                              int32_t* topk_dev, void* stream);

/* ---- bucketing for callers that cannot allocate ---------------------------
 * The Flint blog has no counterpart to this entry point: it serves callers,
 * not the method. It computes what flint_moe_bucket computes, offsets_dev[E+1]
 * and perm_dev[T*k] from idx_dev[T][k] (experts 0..E-1), without a handle and
 * without allocating anything. flint_moe_create allocates a workspace with
 * cudaMalloc; some callers cannot allocate where they need this step: a
 * process whose device memory is already reserved by another allocator (a
 * framework's caching pool), a plugin whose host runtime forbids allocating
 * outside its own allocator, or a loop that cannot afford cudaMalloc's
 * implicit device synchronisation. Its scratch is one static device array of
 * 256 KiB inside the library, which every GPU that loads the library holds
 * until the process exits. Runs on the current device.
 * Limits: 1 <= E <= 256, 1 <= k <= 8, T*k <= 524288; larger sizes return
 * FLINT_EINVAL and enqueue nothing. T == 0 is a no-op.
 * The first call on a device looks up the array's device address (once per
 * device and context, under a lock; again after cudaDeviceReset): make that
 * first call before any stream capture.
 * All calls share the array, so calls that overlap on the GPU race and
 * corrupt each other's results. Expert indices outside 0..E-1 are dropped and
 * nothing reports them (there is no status word): a caller that cannot rule
 * them out checks offsets_dev[E] == T*k, which fails exactly when some were
 * dropped; perm_dev[offsets_dev[E] .. T*k-1] is then left unwritten. */
FLINT_API flint_status flint_moe_bucket_noalloc(const int32_t* idx_dev, int T, int k, int E,
                                                int32_t* offsets_dev, int32_t* perm_dev, void* stream);

/* ---- measurement hooks ---------------------------------------------------- */

/* Dense block-scaled FP4 tensor-core throughput of the current device, the
 * denominator of the FP4 roofline fractions. Every SM runs iters x 4
 * back-to-back tcgen05.mma kind::mxf4nvf4 (scale_vec::4X) of M = 128, N = n
 * (128 or 256), K = 64 on operands resident in shared and tensor memory, one
 * CTA per SM; the timed launch follows one short untimed launch. Writes the
 * launch's CUDA-event time to *ms and the FLOPs it performed (2*M*N*K per MMA)
 * to *flops. Synchronous; allocates a 4-byte status word. Errors:
 * FLINT_EINVAL (n, iters outside 1..2^24, NULL), FLINT_ECUDA, FLINT_ETIMEOUT
 * (the bounded wait for the MMAs gave up). The Flint blog has no counterpart:
 * it is measurement infrastructure. */
FLINT_API flint_status flint_moe_probe_fp4_peak(int n, int iters, float* ms, double* flops);

/* Run one kernel whose bounded wait is made to run out, with the given limit
 * of polls (1 .. 2^20): kind 0 waits on an mbarrier that never completes,
 * kind 1 on a grid barrier (cooperative launch of 2 CTAs) that one CTA never
 * reaches. The kernel records FLINT_ETIMEOUT in the handle's status word and
 * returns; nothing hangs and no copy is in flight. flint_moe_status then
 * reports FLINT_ETIMEOUT and puts the handle's barrier counters back to their
 * idle state, after which the handle is usable. A check of the failure path
 * of every bounded wait in the kernels; the blog has no counterpart.
 * Asynchronous on `stream`. FLINT_EINVAL on bad arguments. */
FLINT_API flint_status flint_moe_debug_wait_timeout(flint_moe* h, int kind, uint32_t spin_limit, void* stream);

/* Number of kernels this handle has launched so far (all entry points). */
FLINT_API uint64_t flint_moe_launch_count(const flint_moe* h);

/* Kernels one single-layer flint_moe_forward of T tokens launches: 1 when the
 * single-launch decode kernel serves T (T <= 2 with one shared expert, if its
 * shared-memory plan fits), otherwise the multi-kernel count. -1 on bad
 * arguments. The single-launch path can be switched off for a handle by
 * setting the environment variable FLINT_MOE_FUSED_DECODE=0 before
 * flint_moe_create. */
FLINT_API int flint_moe_forward_launches(const flint_moe* h, int T);

/* Number of phases flint_moe_profile_end reports. */
#define FLINT_PROFILE_PHASES 5

/* Start recording CUDA events on the caller's stream between the kernels of
 * the next max_forwards single-layer forwards. Phases: 0 router, top-k and
 * bucketing; 1 expert gate/up; 2 expert down projection (and, on the
 * 16-bit-activation path, the combine); 3 activation quantisation (FP4 path:
 * plan, x and h quantisers); 4 output cast and clear of the fp32 sum (FP4
 * path). The single-launch decode kernel counts entirely as phase 0. Phases a
 * path does not have read 0. Allocates the events; FLINT_EINVAL if
 * max_forwards < 1. */
FLINT_API flint_status flint_moe_profile_begin(flint_moe* h, int max_forwards);

/* Wait for the recorded forwards, write the summed duration of each phase in
 * milliseconds to phase_ms[0 .. FLINT_PROFILE_PHASES-1] and the number of
 * recorded forwards to *n_forwards, then free the events and stop recording. */
FLINT_API flint_status flint_moe_profile_end(flint_moe* h, float* phase_ms, int* n_forwards);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_MOE_H */
