// C ABI of the layer: handle, weight loading, forward orchestration.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/flint_moe.h"
#include "kernels.cuh"

using flint::LayerDev;
using flint::Shape;
using flint::Workspace;

struct flint_moe {
    Shape s;
    int n_layers = 0;
    int device = 0;
    std::vector<LayerDev> layers;
    Workspace ws{};
    void* ws_base = nullptr;
    size_t ws_bytes = 0;
    size_t weight_bytes = 0;
    cudaStream_t load_stream = nullptr;
    uint64_t launches = 0;
    int n_sms = 0;
    bool fused = true;           // single-launch decode for T <= kFusedMaxT
    bool stack = true;           // the whole decode stack in one launch (T <= kFusedMaxT)
    flint::StackLayer* stack_table = nullptr;   // [n_layers] device table of the layers' pointers
    bool prefill = true;         // tensor-core (tcgen05) kernels for large T
    bool fp4_experts = false;    // block-scaled FP4 expert GEMMs for T > kSmallT
    void* pws = nullptr;         // their workspace (swizzled activation tiles, h, fp32 sums)
    size_t pws_bytes = 0;
    // events of profiled forwards: kProfMarks per forward (see prof_record)
    std::vector<cudaEvent_t> prof_events;
    int prof_max = 0, prof_n = 0;
    // the 4-bit output head (tiled NVFP4) and its sampler's scratch
    int head_vocab = 0;
    float head_tscale = 0.f;
    uint8_t* head_codes = nullptr;
    uint8_t* head_scales = nullptr;
    void* head_scratch = nullptr;
    flint::HeadScratch head_hs{};
};

namespace {

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        ok = (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

flint_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FLINT_OK;
    if (e == cudaErrorMemoryAllocation) return FLINT_ENOMEM;
    return FLINT_ECUDA;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

void free_layer(LayerDev& L) {
    cudaFree(L.router_hi);
    cudaFree(L.router_lo);
    cudaFree(L.router);
    cudaFree(L.bias);
    cudaFree(L.codes);
    cudaFree(L.scales);
    cudaFree(L.tscale);
    cudaFree(L.prefill);
    cudaFree(L.router_t);
    L = LayerDev{};
}

flint_status validate_config(const flint_moe_config* c) {
    if (c == nullptr) return FLINT_EINVAL;
    if (c->d < 128 || c->d > 4096 || c->d % 128 != 0) return FLINT_EINVAL;
    if (c->f < 128 || c->f > 4096 || c->f % 128 != 0) return FLINT_EINVAL;
    if (c->n_experts < 32 || c->n_experts > 256 || c->n_experts % 32 != 0) return FLINT_EINVAL;
    if (c->top_k < 1 || c->top_k > 8 || c->top_k > c->n_experts) return FLINT_EINVAL;
    if (c->n_shared != 0 && c->n_shared != 1) return FLINT_EINVAL;
    if (c->wfmt != FLINT_W_NVFP4 && c->wfmt != FLINT_W_Q4_1) return FLINT_EINVAL;
    if (c->max_tokens < 1 || c->max_tokens > 65536) return FLINT_EINVAL;
    if (c->n_layers < 1 || c->n_layers > 4096) return FLINT_EINVAL;
    if (c->device < 0) return FLINT_EINVAL;
    return FLINT_OK;
}

// Carve the workspace out of one allocation.
struct Carver {
    char* base;
    size_t off = 0;
    template <class T>
    T* take(size_t count) {
        off = align_up(off, 256);
        T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
        off += count * sizeof(T);
        return p;
    }
};

Workspace carve(const Shape& s, char* base, size_t* total) {
    Carver cv{base};
    Workspace w{};
    const size_t Tm = s.max_tokens;
    const size_t P = (size_t)s.positions(s.max_tokens);
    const size_t n_chunks = (Tm * s.k + flint::kBucketChunk - 1) / flint::kBucketChunk;
    w.logits = cv.take<float>(Tm * s.E);
    w.idx = cv.take<int>(Tm * s.k);
    w.w = cv.take<float>(Tm * s.k);
    w.perm = cv.take<int>(Tm * s.k);
    w.inv = cv.take<int>(Tm * s.k);
    w.offsets = cv.take<int>(s.E + 1);
    w.ecount = cv.take<int>((size_t)s.E * flint::kEcountStride);
    w.slot_expert = cv.take<int>(s.E + 1);
    w.slot_off = cv.take<int>(s.E + 1);
    w.slot_cnt = cv.take<int>(s.E + 1);
    w.meta = cv.take<int>(8);
    w.x16 = cv.take<__half>(Tm * s.d);
    w.xinv = cv.take<float>(Tm);
    w.hf = cv.take<float>(P * s.f);
    w.hamax = cv.take<uint32_t>(P);
    w.yw = cv.take<float>(P * s.d);
    w.chunk_hist = cv.take<int>(n_chunks * s.E);
    w.counters = cv.take<uint32_t>(flint::kCounters);
    w.gbar = cv.take<uint32_t>(64);
    w.dbg = cv.take<uint32_t>(64);
    w.gbar8 = cv.take<unsigned long long>((size_t)flint::kGridGroups * flint::kGridGroupStride);
    w.racc = cv.take<unsigned long long>((size_t)2 * flint::kRaccCopies * flint::kFusedMaxT * s.E);
    w.rnf = cv.take<uint32_t>((size_t)2 * flint::kRaccCopies * flint::kFusedMaxT * s.E);
    w.status = cv.take<uint32_t>(1);
    *total = align_up(cv.off, 256);
    return w;
}

bool finite_f32(const float* p, size_t n) {
    for (size_t i = 0; i < n; ++i)
        if (!isfinite(p[i])) return false;
    return true;
}

flint_status check_forward_args(flint_moe* h, int layer, const void* a, const void* b, int T) {
    if (h == nullptr) return FLINT_EINVAL;
    if (layer < 0 || layer >= h->n_layers) return FLINT_EINVAL;
    if (T < 0 || T > h->s.max_tokens) return FLINT_EINVAL;
    if (T > 0) {
        if (a == nullptr || !aligned16(a)) return FLINT_EINVAL;
        if (b != nullptr && !aligned16(b)) return FLINT_EINVAL;
    }
    if (!h->layers[layer].loaded) return FLINT_ESTATE;
    return FLINT_OK;
}

void prof_free(flint_moe* h) {
    for (cudaEvent_t ev : h->prof_events) cudaEventDestroy(ev);
    h->prof_events.clear();
    h->prof_max = h->prof_n = 0;
}

// Marks of one profiled forward: 0 start, 1 routing done, 2 activations
// quantised, 3 gate/up done, 4 h quantised, 5 down projection done, 6 output
// written. A path without a step records its two marks back to back.
// Phases: router 1-0, gate/up 3-2, down 5-4, quantisation (2-1)+(4-3), cast 6-5.
constexpr int kProfMarks = 7;

cudaEvent_t* prof_marks(flint_moe* h) {
    return h->prof_n < h->prof_max ? &h->prof_events[(size_t)h->prof_n * kProfMarks] : nullptr;
}
void prof_record(flint_moe* h, int mark, cudaStream_t st) {
    if (h->prof_n < h->prof_max) cudaEventRecord(h->prof_events[(size_t)h->prof_n * kProfMarks + mark], st);
}
void prof_next(flint_moe* h) {
    if (h->prof_n < h->prof_max) ++h->prof_n;
}

cudaError_t run_layer(flint_moe* h, int layer, const __nv_bfloat16* x, int T, __nv_bfloat16* out,
                      const __nv_bfloat16* residual, cudaStream_t st, const LayerDev* next = nullptr) {
    const LayerDev& L = h->layers[layer];
    int n = 0;
    int n_slots = 0, offs[10];
    if (h->fused && flint::fused_smem_bytes(h->s, T, h->n_sms, &n_slots, offs) != 0) {
        flint::FusedScratch fs{h->ws.logits, h->ws.hf, h->ws.gbar, h->ws.status};
        prof_record(h, 0, st);
        cudaError_t e = flint::launch_decode_fused(h->s, L, x, T, out, residual, fs, h->n_sms, st, next);
        for (int k = 1; k < kProfMarks; ++k) prof_record(h, k, st);
        prof_next(h);
        h->launches += 1;
        return e;
    }
    if (T > flint::kSmallT && h->fp4_experts && L.prefill != nullptr) {
        prof_record(h, 0, st);
        cudaError_t e = flint::launch_router_fp4(h->s, L, x, T, h->ws, st, &n);
        prof_record(h, 1, st);
        if (e == cudaSuccess)
            e = flint::launch_prefill_experts(h->s, L, x, T, h->ws, static_cast<uint8_t*>(h->pws), h->s.max_tokens,
                                              out, residual, st, &n, prof_marks(h) ? prof_marks(h) + 1 : nullptr);
        prof_next(h);
        h->launches += n;
        return e;
    }
    prof_record(h, 0, st);
    cudaError_t e = flint::launch_router(h->s, L, x, T, h->ws, st, &n);
    prof_record(h, 1, st);
    prof_record(h, 2, st);
    if (e == cudaSuccess) e = flint::launch_gateup(h->s, L, T, h->ws, st, &n);
    prof_record(h, 3, st);
    prof_record(h, 4, st);
    if (e == cudaSuccess) e = flint::launch_down(h->s, L, T, h->ws, out, residual, st, &n);
    prof_record(h, 5, st);
    prof_record(h, 6, st);
    prof_next(h);
    h->launches += n;
    return e;
}

}  // namespace

extern "C" {

const char* flint_moe_status_string(flint_status s) {
    switch (s) {
        case FLINT_OK: return "ok";
        case FLINT_EINVAL: return "invalid argument";
        case FLINT_ENOMEM: return "out of device memory";
        case FLINT_ECUDA: return "CUDA error";
        case FLINT_ESTATE: return "layer weights not loaded";
        case FLINT_ETIMEOUT: return "device wait timed out";
        case FLINT_ENOTIMPL: return "not implemented";
        case FLINT_EDEVICE: return "device reported a data fault";
    }
    return "unknown status";
}

flint_status flint_moe_create(const flint_moe_config* cfg, flint_moe** out) {
    if (out == nullptr) return FLINT_EINVAL;
    *out = nullptr;
    flint_status st = validate_config(cfg);
    if (st != FLINT_OK) return st;
    int n_dev = 0;
    if (cudaGetDeviceCount(&n_dev) != cudaSuccess || cfg->device >= n_dev) return FLINT_EINVAL;
    DeviceGuard guard(cfg->device);
    if (!guard.ok) return FLINT_ECUDA;
    flint_moe* h = new (std::nothrow) flint_moe();
    if (h == nullptr) return FLINT_ENOMEM;
    h->s = Shape{cfg->d, cfg->f, cfg->n_experts, cfg->top_k, cfg->n_shared, cfg->wfmt, cfg->max_tokens};
    h->n_layers = cfg->n_layers;
    h->device = cfg->device;
    if (cudaDeviceGetAttribute(&h->n_sms, cudaDevAttrMultiProcessorCount, cfg->device) != cudaSuccess) {
        delete h;
        return FLINT_ECUDA;
    }
    {
        const char* env = getenv("FLINT_MOE_FUSED_DECODE");
        if (env != nullptr && env[0] == '0') h->fused = false;
    }
    if (h->fused && flint::prepare_decode_fused() != cudaSuccess) h->fused = false;
    {
        const char* env = getenv("FLINT_MOE_STACK_KERNEL");
        // the one-launch stack kernel unless FLINT_MOE_STACK_KERNEL=0 (then a
        // stack runs one single-layer launch per layer)
        h->stack = h->fused && !(env != nullptr && env[0] == '0');
    }
    {
        const char* env = getenv("FLINT_MOE_TCGEN05_PREFILL");
        if (env != nullptr && env[0] == '0') h->prefill = false;
    }
    if (h->prefill && flint::prepare_prefill() != cudaSuccess) h->prefill = false;
    {
        const char* env = getenv("FLINT_MOE_FP4_EXPERTS");
        h->fp4_experts = h->prefill && !(env != nullptr && env[0] == '0') && cfg->max_tokens > flint::kSmallT &&
                         flint::prefill_fp4_supported(h->s) && flint::prepare_prefill_fp4() == cudaSuccess;
    }
    if (flint::prepare_router() != cudaSuccess || flint::prepare_experts() != cudaSuccess) {
        delete h;
        return FLINT_ECUDA;
    }
    h->layers.resize(cfg->n_layers);
    size_t total = 0;
    carve(h->s, nullptr, &total);
    cudaError_t e = cudaMalloc(&h->ws_base, total);
    if (e != cudaSuccess) {
        delete h;
        return cuda_status(e);
    }
    h->ws_bytes = total;
    h->ws = carve(h->s, static_cast<char*>(h->ws_base), &total);
    if (h->fp4_experts) {
        h->pws_bytes = flint::prefill_workspace_bytes(h->s, cfg->max_tokens);
        e = cudaMalloc(&h->pws, h->pws_bytes);
        if (e == cudaSuccess) e = cudaMemset(h->pws, 0, h->pws_bytes);
        if (e != cudaSuccess) {
            cudaFree(h->pws);
            cudaFree(h->ws_base);
            delete h;
            return cuda_status(e);
        }
    }
    e = cudaMemset(h->ws_base, 0, total);
    if (e == cudaSuccess && h->stack) {
        e = cudaMalloc(&h->stack_table, (size_t)cfg->n_layers * sizeof(flint::StackLayer));
        if (e == cudaSuccess) e = cudaMemset(h->stack_table, 0, (size_t)cfg->n_layers * sizeof(flint::StackLayer));
    }
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->load_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(h->stack_table);
        cudaFree(h->pws);
        cudaFree(h->ws_base);
        delete h;
        return cuda_status(e);
    }
    *out = h;
    return FLINT_OK;
}

flint_status flint_moe_load_weights(flint_moe* h, int layer, const flint_moe_weights* w) {
    if (h == nullptr || w == nullptr) return FLINT_EINVAL;
    if (layer < 0 || layer >= h->n_layers) return FLINT_EINVAL;
    if (w->router == nullptr || w->codes == nullptr || w->scales == nullptr) return FLINT_EINVAL;
    const Shape& s = h->s;
    if (s.wfmt == FLINT_W_NVFP4 && w->tensor_scale == nullptr) return FLINT_EINVAL;
    const int n_slots = s.n_slots();
    const size_t cpm = s.codes_per_matrix(), spm = s.scales_per_matrix();
    const size_t n_codes = (size_t)n_slots * 3 * cpm, n_scales = (size_t)n_slots * 3 * spm;
    // host-side validation
    if (!finite_f32(w->router, (size_t)s.E * s.d)) return FLINT_EINVAL;
    if (w->router_bias && !finite_f32(w->router_bias, s.E)) return FLINT_EINVAL;
    if (s.wfmt == FLINT_W_NVFP4) {
        if (!finite_f32(w->tensor_scale, (size_t)n_slots * 3)) return FLINT_EINVAL;
        for (size_t i = 0; i < n_scales; ++i)
            if (w->scales[i] > 0x7E) return FLINT_EINVAL;   // sign bit set, or NaN
    } else {
        for (size_t i = 0; i < n_scales; i += 2) {
            const uint16_t v = (uint16_t)(w->scales[i] | (w->scales[i + 1] << 8));
            if (((v >> 10) & 0x1f) == 0x1f) return FLINT_EINVAL;   // inf or NaN
        }
    }
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    LayerDev& L = h->layers[layer];
    cudaError_t e = cudaSuccess;
    // the bf16 hi/lo split of the router feeds only the tensor-core router,
    // which serves T > kSmallT: handles that never see such T do not keep it
    const bool want_split = h->prefill && s.max_tokens > flint::kSmallT && flint::router_umma_supported(s);
    if (L.codes == nullptr) {
        e = cudaMalloc(&L.router, (size_t)s.E * s.d * sizeof(float));
        if (e == cudaSuccess) e = cudaMalloc(&L.bias, (size_t)s.E * sizeof(float));
        if (e == cudaSuccess) e = cudaMalloc(&L.codes, n_codes);
        if (e == cudaSuccess) e = cudaMalloc(&L.scales, n_scales);
        if (e == cudaSuccess && want_split) e = cudaMalloc(&L.router_hi, (size_t)s.E * s.d * 2);
        if (e == cudaSuccess && want_split) e = cudaMalloc(&L.router_lo, (size_t)s.E * s.d * 2);
        if (e == cudaSuccess) e = cudaMalloc(&L.tscale, flint::tscale_bytes(s));
        if (e == cudaSuccess) e = cudaMemset(L.tscale, 0, flint::tscale_bytes(s));
        if (e == cudaSuccess && h->fp4_experts) e = cudaMalloc(&L.prefill, flint::prefill_weight_bytes(s));
        if (e == cudaSuccess && h->stack) e = cudaMalloc(&L.router_t, (size_t)s.E * s.d * sizeof(float));
        if (e != cudaSuccess) {
            free_layer(L);
            return cuda_status(e);
        }
        h->weight_bytes += (size_t)s.E * s.d * 4 + (size_t)s.E * 4 + n_codes + n_scales + flint::tscale_bytes(s);
        if (L.router_hi != nullptr) h->weight_bytes += (size_t)s.E * s.d * 4;
        if (L.router_t != nullptr) h->weight_bytes += (size_t)s.E * s.d * 4;
        if (L.prefill != nullptr) h->weight_bytes += flint::prefill_weight_bytes(s);
    }
    L.loaded = false;
    uint8_t* stage = nullptr;
    e = cudaMalloc(&stage, n_codes + n_scales);
    if (e != cudaSuccess) return cuda_status(e);
    cudaStream_t st = h->load_stream;
    e = cudaMemcpyAsync(L.router, w->router, (size_t)s.E * s.d * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) {
        if (w->router_bias)
            e = cudaMemcpyAsync(L.bias, w->router_bias, (size_t)s.E * sizeof(float), cudaMemcpyHostToDevice, st);
        else
            e = cudaMemsetAsync(L.bias, 0, (size_t)s.E * sizeof(float), st);
    }
    if (e == cudaSuccess) {
        if (s.wfmt == FLINT_W_NVFP4) {
            e = cudaMemcpyAsync(L.tscale, w->tensor_scale, (size_t)n_slots * 3 * sizeof(float),
                                cudaMemcpyHostToDevice, st);
        } else {
            std::vector<float> ones((size_t)n_slots * 3, 1.0f);
            e = cudaMemcpyAsync(L.tscale, ones.data(), ones.size() * sizeof(float), cudaMemcpyHostToDevice, st);
            if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        }
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(stage, w->codes, n_codes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(stage + n_codes, w->scales, n_scales, cudaMemcpyHostToDevice, st);
    for (int sl = 0; sl < n_slots && e == cudaSuccess; ++sl) {
        for (int m = 0; m < 3 && e == cudaSuccess; ++m) {
            const int R = m < 2 ? s.f : s.d, K = m < 2 ? s.d : s.f;
            const size_t mi = (size_t)sl * 3 + m;
            e = flint::launch_repack_matrix(stage + mi * cpm, stage + n_codes + mi * spm, L.codes + mi * cpm,
                                            L.scales + mi * spm, R, K, s.wfmt, st);
        }
    }
    if (e == cudaSuccess && L.prefill != nullptr)
        e = flint::pack_prefill_weights(s, stage, stage + n_codes, L.prefill, st);
    if (e == cudaSuccess && L.router_hi != nullptr)
        e = flint::split_router(L.router, L.router_hi, L.router_lo, (size_t)s.E * s.d, st);
    if (e == cudaSuccess && L.router_t != nullptr) e = flint::transpose_router(L.router, L.router_t, s.E, s.d, st);
    if (e == cudaSuccess && h->stack_table != nullptr) {
        const flint::StackLayer sl{L.codes, L.scales, L.tscale, L.router_t, L.bias};
        e = cudaMemcpyAsync(h->stack_table + layer, &sl, sizeof(sl), cudaMemcpyHostToDevice, st);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(stage);
    if (e != cudaSuccess) return cuda_status(e);
    L.umma_router = L.router_hi != nullptr && flint::make_tmap_bf16(&L.tmap_router_hi, L.router_hi, s.E, s.d) &&
                    flint::make_tmap_bf16(&L.tmap_router_lo, L.router_lo, s.E, s.d);
    L.loaded = true;
    return FLINT_OK;
}

flint_status flint_moe_forward(flint_moe* h, int layer, const void* hidden_dev, int T, void* out_dev,
                               void* stream) {
    flint_status st = check_forward_args(h, layer, hidden_dev, out_dev, T);
    if (st != FLINT_OK) return st;
    if (T > 0 && out_dev == nullptr) return FLINT_EINVAL;
    if (T == 0) return FLINT_OK;
    const char* x0 = static_cast<const char*>(hidden_dev);
    const char* o0 = static_cast<const char*>(out_dev);
    const size_t bytes = (size_t)T * h->s.d * 2;
    if (x0 < o0 + bytes && o0 < x0 + bytes) return FLINT_EINVAL;   // overlap
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    cudaError_t e = run_layer(h, layer, static_cast<const __nv_bfloat16*>(hidden_dev), T,
                              static_cast<__nv_bfloat16*>(out_dev), nullptr, (cudaStream_t)stream);
    return cuda_status(e);
}

flint_status flint_moe_forward_stack(flint_moe* h, int layer0, int n_layers, void* hidden_dev, int T,
                                     void* stream) {
    if (h == nullptr || n_layers < 0) return FLINT_EINVAL;
    if (layer0 < 0 || layer0 + n_layers > h->n_layers) return FLINT_EINVAL;
    for (int l = layer0; l < layer0 + n_layers; ++l) {
        flint_status st = check_forward_args(h, l, hidden_dev, nullptr, T);
        if (st != FLINT_OK) return st;
    }
    if (T == 0 || n_layers == 0) return FLINT_OK;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    __nv_bfloat16* x = static_cast<__nv_bfloat16*>(hidden_dev);
    if (h->stack && T <= flint::kFusedMaxT && flint::stack_smem_bytes(h->s, T, h->n_sms) != 0) {
        // every layer in one persistent launch
        flint::FusedScratch fs{h->ws.logits, h->ws.hf, h->ws.gbar, h->ws.status};
        const cudaError_t e = flint::launch_decode_stack(h->s, h->stack_table + layer0, n_layers, x, T, fs,
                                                         h->ws.gbar8, h->ws.racc, h->ws.rnf, h->n_sms,
                                                         (cudaStream_t)stream);
        if (e == cudaSuccess) h->launches += 1;
        return cuda_status(e);
    }
    for (int l = layer0; l < layer0 + n_layers; ++l) {
        const LayerDev* next = (l + 1 < layer0 + n_layers && h->layers[l + 1].loaded) ? &h->layers[l + 1] : nullptr;
        cudaError_t e = run_layer(h, l, x, T, x, x, (cudaStream_t)stream, next);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return FLINT_OK;
}

void flint_moe_destroy(flint_moe* h) {
    if (h == nullptr) return;
    {
        DeviceGuard guard(h->device);
        cudaDeviceSynchronize();
        for (auto& L : h->layers) free_layer(L);
        prof_free(h);
        cudaFree(h->head_codes);
        cudaFree(h->head_scales);
        cudaFree(h->head_scratch);
        cudaFree(h->ws_base);
        cudaFree(h->pws);
        cudaFree(h->stack_table);
        if (h->load_stream) cudaStreamDestroy(h->load_stream);
    }
    delete h;
}

// ---------------------------------------------------------------------------
// The 4-bit output head and its sampler
// ---------------------------------------------------------------------------

flint_status flint_moe_load_lm_head(flint_moe* h, int vocab, const void* codes, const void* scales,
                                    float tensor_scale) {
    if (h == nullptr || codes == nullptr || scales == nullptr) return FLINT_EINVAL;
    if (vocab <= 0 || vocab % 8 != 0 || h->s.d > flint::kHeadMaxD || !isfinite(tensor_scale)) return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return FLINT_ECUDA;
    cudaFree(h->head_codes);
    cudaFree(h->head_scales);
    cudaFree(h->head_scratch);
    h->head_codes = h->head_scales = nullptr;
    h->head_scratch = nullptr;
    h->head_vocab = 0;
    const size_t n_codes = (size_t)vocab * h->s.d / 2, n_scales = (size_t)vocab * h->s.d / 16;
    const int parts = flint::head_sample_parts(vocab);
    const size_t n_cand = (size_t)flint::kHeadMaxT * parts * 32;
    uint8_t* stage = nullptr;
    e = cudaMalloc(&h->head_codes, n_codes);
    if (e == cudaSuccess) e = cudaMalloc(&h->head_scales, n_scales);
    if (e == cudaSuccess) e = cudaMalloc(&h->head_scratch, n_cand * 8 + flint::kHeadMaxT * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMalloc(&stage, n_codes + n_scales);
    cudaStream_t st = h->load_stream;
    if (e == cudaSuccess) e = cudaMemcpyAsync(stage, codes, n_codes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(stage + n_codes, scales, n_scales, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = flint::launch_repack_matrix(stage, stage + n_codes, h->head_codes, h->head_scales, vocab, h->s.d,
                                        FLINT_W_NVFP4, st);
    if (e == cudaSuccess) {
        auto* base = static_cast<uint8_t*>(h->head_scratch);
        h->head_hs.cand_key = reinterpret_cast<uint32_t*>(base);
        h->head_hs.cand_idx = reinterpret_cast<uint32_t*>(base + n_cand * 4);
        h->head_hs.counters = reinterpret_cast<unsigned*>(base + n_cand * 8);
        e = cudaMemsetAsync(h->head_hs.counters, 0, flint::kHeadMaxT * sizeof(unsigned), st);
    }
    if (e == cudaSuccess) e = flint::prepare_head();
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(stage);
    if (e != cudaSuccess) {
        cudaFree(h->head_codes);
        cudaFree(h->head_scales);
        cudaFree(h->head_scratch);
        h->head_codes = h->head_scales = nullptr;
        h->head_scratch = nullptr;
        return cuda_status(e);
    }
    h->head_vocab = vocab;
    h->head_tscale = tensor_scale;
    return FLINT_OK;
}

flint_status flint_moe_lm_head(flint_moe* h, const void* hidden_dev, int T, float* logits_dev, void* stream) {
    if (h == nullptr || T < 0 || T > flint::kHeadMaxT) return FLINT_EINVAL;
    if (h->head_vocab == 0) return FLINT_ESTATE;
    if (T == 0) return FLINT_OK;
    if (hidden_dev == nullptr || logits_dev == nullptr || !aligned16(hidden_dev) || !aligned16(logits_dev))
        return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    const cudaError_t e = flint::launch_head_gemv(h->head_codes, h->head_scales, h->head_tscale,
                                                  static_cast<const __nv_bfloat16*>(hidden_dev), T, h->s.d,
                                                  h->head_vocab, logits_dev, h->n_sms, (cudaStream_t)stream);
    if (e == cudaSuccess) h->launches += 1;
    return cuda_status(e);
}

flint_status flint_moe_sample(flint_moe* h, const float* logits_dev, int T, float temperature, int top_k,
                              float top_p, const float* u_dev, int32_t* tokens_dev, int32_t* topk_dev,
                              void* stream) {
    if (h == nullptr || T < 0 || T > flint::kHeadMaxT) return FLINT_EINVAL;
    if (h->head_vocab == 0) return FLINT_ESTATE;
    if (!isfinite(temperature) || !(top_p > 0.f && top_p <= 1.f)) return FLINT_EINVAL;
    if (!flint::head_sample_supported(h->head_vocab, top_k)) return FLINT_EINVAL;
    if (T == 0) return FLINT_OK;
    if (logits_dev == nullptr || u_dev == nullptr || tokens_dev == nullptr) return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    const cudaError_t e = flint::launch_head_sample(logits_dev, T, h->head_vocab, temperature, top_k, top_p, u_dev,
                                                    tokens_dev, topk_dev, h->head_hs, h->ws.status,
                                                    (cudaStream_t)stream);
    if (e == cudaSuccess) h->launches += 1;
    return cuda_status(e);
}

flint_status flint_moe_status(flint_moe* h) {
    if (h == nullptr) return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return FLINT_ECUDA;
    uint32_t v = 0;
    e = cudaMemcpy(&v, h->ws.status, sizeof(v), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->ws.status, 0, sizeof(v));
    if (e == cudaSuccess && (v & flint::kStatusTimeout)) {
        // a kernel left a barrier early: its arrival counters may be off, so
        // put every counter back to its between-launches value (zero); the
        // device is idle here
        e = cudaMemset(h->ws.gbar, 0, 64 * sizeof(uint32_t));
        if (e == cudaSuccess) e = cudaMemset(h->ws.counters, 0, flint::kCounters * sizeof(uint32_t));
        if (e == cudaSuccess && h->head_hs.counters != nullptr)
            e = cudaMemset(h->head_hs.counters, 0, flint::kHeadMaxT * sizeof(unsigned));
        // the decode stack's router accumulators are zero between launches
        const size_t nacc = (size_t)2 * flint::kRaccCopies * flint::kFusedMaxT * h->s.E;
        if (e == cudaSuccess) e = cudaMemset(h->ws.racc, 0, nacc * 8);
        if (e == cudaSuccess) e = cudaMemset(h->ws.rnf, 0, nacc * 4);
        if (e == cudaSuccess)
            e = cudaMemset(h->ws.gbar8, 0, (size_t)flint::kGridGroups * flint::kGridGroupStride * 8);
        if (e == cudaSuccess) e = cudaMemset(h->ws.ecount, 0, (size_t)h->s.E * flint::kEcountStride * sizeof(int));
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return FLINT_ECUDA;
    if (v & flint::kStatusTimeout) return FLINT_ETIMEOUT;
    if (v != 0) return FLINT_EDEVICE;
    return FLINT_OK;
}

flint_status flint_moe_router(flint_moe* h, int layer, const void* hidden_dev, int T, float* logits_dev,
                              int32_t* idx_dev, float* w_dev, void* stream) {
    flint_status st = check_forward_args(h, layer, hidden_dev, nullptr, T);
    if (st != FLINT_OK) return st;
    if (T == 0) return FLINT_OK;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const LayerDev& L = h->layers[layer];
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(hidden_dev);
    int n = 0;
    cudaError_t e = flint::launch_router(h->s, L, x, T, h->ws, s, &n);
    h->launches += n;
    if (e == cudaSuccess && logits_dev)
        e = cudaMemcpyAsync(logits_dev, h->ws.logits, (size_t)T * h->s.E * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && idx_dev)
        e = cudaMemcpyAsync(idx_dev, h->ws.idx, (size_t)T * h->s.k * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && w_dev)
        e = cudaMemcpyAsync(w_dev, h->ws.w, (size_t)T * h->s.k * 4, cudaMemcpyDeviceToDevice, s);
    return cuda_status(e);
}

flint_status flint_moe_topk(const float* logits_dev, int T, int E, int k, int32_t* idx_dev, float* w_dev,
                            void* stream) {
    if (T < 0 || E < 32 || E > 256 || E % 32 != 0 || k < 1 || k > 8 || k > E) return FLINT_EINVAL;
    if (T == 0) return FLINT_OK;
    if (logits_dev == nullptr || idx_dev == nullptr) return FLINT_EINVAL;
    return cuda_status(flint::launch_topk(logits_dev, T, E, k, idx_dev, w_dev, (cudaStream_t)stream));
}

flint_status flint_moe_bucket(flint_moe* h, const int32_t* idx_dev, int T, int32_t* offsets_dev,
                              int32_t* perm_dev, void* stream) {
    if (h == nullptr || T < 0 || T > h->s.max_tokens) return FLINT_EINVAL;
    if (T == 0) return FLINT_OK;
    if (idx_dev == nullptr || offsets_dev == nullptr || perm_dev == nullptr) return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int n = 0;
    cudaError_t e = flint::launch_bucket(h->s, idx_dev, T, h->ws, s, &n);
    h->launches += n;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(offsets_dev, h->ws.offsets, (size_t)(h->s.E + 1) * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(perm_dev, h->ws.perm, (size_t)T * h->s.k * 4, cudaMemcpyDeviceToDevice, s);
    return cuda_status(e);
}

flint_status flint_moe_dequant(flint_moe* h, int layer, int expert, int mat, float* out_dev, void* stream) {
    if (h == nullptr || out_dev == nullptr) return FLINT_EINVAL;
    if (layer < 0 || layer >= h->n_layers) return FLINT_EINVAL;
    if (expert < 0 || expert >= h->s.n_slots() || mat < 0 || mat > 2) return FLINT_EINVAL;
    if (!h->layers[layer].loaded) return FLINT_ESTATE;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    const Shape& s = h->s;
    const LayerDev& L = h->layers[layer];
    const int R = mat < 2 ? s.f : s.d, K = mat < 2 ? s.d : s.f;
    const size_t mi = (size_t)expert * 3 + mat;
    cudaError_t e = flint::launch_dequant_matrix(L.codes + mi * s.codes_per_matrix(),
                                                 L.scales + mi * s.scales_per_matrix(), 1.0f,
                                                 s.wfmt == FLINT_W_NVFP4 ? L.tscale + mi : nullptr, R, K,
                                                 s.wfmt, out_dev, (cudaStream_t)stream);
    return cuda_status(e);
}

flint_status flint_moe_debug_wait_timeout(flint_moe* h, int kind, uint32_t spin_limit, void* stream) {
    if (h == nullptr || (kind != 0 && kind != 1) || spin_limit < 1 || spin_limit > (1u << 20)) return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    const cudaError_t e = flint::launch_wait_timeout(kind, spin_limit, reinterpret_cast<unsigned long long*>(h->ws.dbg),
                                                     h->ws.status, (cudaStream_t)stream);
    if (e == cudaSuccess) h->launches += 1;
    return cuda_status(e);
}

flint_status flint_moe_probe_fp4_peak(int n, int iters, float* ms, double* flops) {
    if ((n != 128 && n != 256) || iters < 1 || iters > (1 << 24) || ms == nullptr || flops == nullptr)
        return FLINT_EINVAL;
    int dev = 0, n_sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_ECUDA;
    if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FLINT_ECUDA;
    uint32_t* status = nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e = cudaMalloc(&status, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(status, 0, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    // one short launch first (code, clocks), then the timed one
    if (e == cudaSuccess) e = flint::launch_fp4_peak(n, iters / 16 + 1, n_sms, status, st);
    if (e == cudaSuccess) e = cudaEventRecord(e0, st);
    if (e == cudaSuccess) e = flint::launch_fp4_peak(n, iters, n_sms, status, st);
    if (e == cudaSuccess) e = cudaEventRecord(e1, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
    uint32_t hs = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&hs, status, sizeof(hs), cudaMemcpyDeviceToHost);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (st) cudaStreamDestroy(st);
    cudaFree(status);
    if (e != cudaSuccess) return cuda_status(e);
    if (hs != 0) return FLINT_ETIMEOUT;
    *ms = t;
    // per MMA: M = 128, N = n, K = 64; four MMAs per iteration on every SM
    *flops = 2.0 * 128.0 * n * 64.0 * 4.0 * (double)iters * n_sms;
    return FLINT_OK;
}

size_t flint_moe_device_bytes(const flint_moe* h) {
    if (h == nullptr) return 0;
    return h->ws_bytes + h->pws_bytes + h->weight_bytes;
}

uint64_t flint_moe_launch_count(const flint_moe* h) { return h ? h->launches : 0; }

int flint_moe_tensor_core_plan(const flint_moe* h, int layer, int T) {
    if (h == nullptr || layer < 0 || layer >= h->n_layers || T < 0 || T > h->s.max_tokens) return -1;
    const LayerDev& L = h->layers[layer];
    int plan = 0;
    if (T > flint::kSmallT && L.loaded && L.umma_router) plan |= 1;
    if (T > flint::kSmallT && L.loaded && h->fp4_experts && L.prefill != nullptr) plan |= 2;
    return plan;
}

int flint_moe_forward_launches(const flint_moe* h, int T) {
    if (h == nullptr || T < 0 || T > h->s.max_tokens) return -1;
    if (T == 0) return 0;
    int n_slots = 0, offs[10];
    if (h->fused && flint::fused_smem_bytes(h->s, T, h->n_sms, &n_slots, offs) != 0) return 1;
    const int router = flint::router_fused(h->s, T) ? 1 : 2 + 3;
    if (T > flint::kSmallT && h->fp4_experts) return 2 + 6;   // logits, top-k and ranks; 6 expert-path kernels
    return router + flint::expert_launches(h->s, T);
}

flint_status flint_moe_profile_begin(flint_moe* h, int max_forwards) {
    if (h == nullptr || max_forwards < 1 || max_forwards > (1 << 22)) return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    prof_free(h);
    h->prof_events.resize((size_t)max_forwards * kProfMarks);
    for (size_t i = 0; i < h->prof_events.size(); ++i) {
        if (cudaEventCreate(&h->prof_events[i]) != cudaSuccess) {
            h->prof_events.resize(i);
            prof_free(h);
            return FLINT_ECUDA;
        }
    }
    h->prof_max = max_forwards;
    h->prof_n = 0;
    return FLINT_OK;
}

flint_status flint_moe_profile_end(flint_moe* h, float* phase_ms, int* n_forwards) {
    if (h == nullptr || phase_ms == nullptr || n_forwards == nullptr) return FLINT_EINVAL;
    DeviceGuard guard(h->device);
    if (!guard.ok) return FLINT_ECUDA;
    // interval i = marks (i, i+1) -> phase
    static const int kPhaseOf[kProfMarks - 1] = {0, 3, 1, 3, 2, 4};
    double acc[FLINT_PROFILE_PHASES] = {0, 0, 0, 0, 0};
    cudaError_t e = cudaSuccess;
    for (int f = 0; f < h->prof_n && e == cudaSuccess; ++f) {
        const cudaEvent_t* ev = &h->prof_events[(size_t)f * kProfMarks];
        e = cudaEventSynchronize(ev[kProfMarks - 1]);
        for (int i = 0; i + 1 < kProfMarks && e == cudaSuccess; ++i) {
            float ms = 0.f;
            e = cudaEventElapsedTime(&ms, ev[i], ev[i + 1]);
            acc[kPhaseOf[i]] += ms;
        }
    }
    for (int p = 0; p < FLINT_PROFILE_PHASES; ++p) phase_ms[p] = (float)acc[p];
    *n_forwards = h->prof_n;
    prof_free(h);
    return cuda_status(e);
}

}  // extern "C"
