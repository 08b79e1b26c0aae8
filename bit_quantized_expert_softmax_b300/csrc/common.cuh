// Device helpers shared by the layer's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace flint {

constexpr int kWarp = 32;
constexpr int kKTile = 128;   // K elements per weight tile (8 mma k16 steps)
constexpr int kRowTile = 8;   // rows per weight tile

// Device status word bits.
constexpr uint32_t kStatusNonFiniteLogit = 1u;
constexpr uint32_t kStatusBadIndex = 2u;
constexpr uint32_t kStatusTimeout = 4u;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// Fragment permutation inside a 128-element K tile.
//
// mma.m16n8k16 gives lane (g = lane/4, c = lane%4) the K positions
// {2c, 2c+1, 2c+8, 2c+9} of every 16-wide step. Activations are stored so that
// one lane's four values of all 8 steps of a tile are contiguous:
//   position p = c*32 + s*4 + j  holds  K index 16*s + {2c, 2c+1, 2c+8, 2c+9}[j]
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int kperm_pos(int k /* 0..127 */) {
    int s = k >> 4, r = k & 15;
    int c = (r & 7) >> 1;
    int j = (r & 1) | ((r >> 3) << 1);
    return c * 32 + s * 4 + j;
}

// ---------------------------------------------------------------------------
// 4-bit and 8-bit float conversions (hardware cvt, exact)
// ---------------------------------------------------------------------------

// Four bytes of packed E2M1 pairs -> four f16x2 (byte i -> r[i]; the low
// nibble goes to the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& r0, uint32_t& r1,
                                                uint32_t& r2, uint32_t& r3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
}

// Two E4M3 bytes (low 16 bits of w) -> f16x2 (low byte -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
    uint32_t r;
    uint16_t v = (uint16_t)(w & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// broadcast the low / high f16 of x to both halves
__device__ __forceinline__ uint32_t bcast_lo(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

// q4_1: byte (two 4-bit q) -> f16x2 {q_lo, q_hi} exactly, via 1024 + q.
__device__ __forceinline__ uint32_t q4x2_to_f16x2(uint32_t byte) {
    uint32_t v = 0x64006400u | (byte & 0xfu) | ((byte & 0xf0u) << 12);
    return hsub2_u(v, 0x64006400u);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// mma.sync m16n8k16, f16 inputs, f32 accumulate (D = A B + D)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

// 2^e as float for e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Power-of-two multiplier that brings a positive amax into [2^14, 2^15):
// values scaled by it fit fp16 with full precision. 1 for amax 0 or non-finite.
__device__ __forceinline__ float f16_range_mult(float amax) {
    uint32_t b = __float_as_uint(amax);
    int ef = (int)((b >> 23) & 0xff);
    if (amax <= 0.0f || ef == 0xff) return 1.0f;
    int e = (ef == 0) ? -126 : ef - 127;   // floor(log2(amax)) for normals
    int m = 14 - e;
    m = m > 126 ? 126 : (m < -126 ? -126 : m);
    return exp2i(m);
}

}  // namespace flint

namespace flint {

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk (TMA, 1-D) copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy completing on an mbarrier. dst, src 16-byte
// aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Bounded wait for an mbarrier phase: at most `limit` polls. Returns false
// (and records a timeout in the status word) if the phase does not complete
// within the limit.
constexpr uint32_t kMbarSpinLimit = 1u << 22;

__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, uint32_t phase, uint32_t* status, uint32_t limit) {
    for (uint32_t it = 0; it < limit; ++it) {
        if (mbar_try_wait(bar, phase)) return true;
    }
    if (status) atomicOr(status, kStatusTimeout);
    return false;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase, uint32_t* status) {
    return mbar_wait_limit(bar, phase, status, kMbarSpinLimit);
}

// A ring of n_stages shared-memory stages, each filled by bulk copies that
// complete on full[stage]; fill number i (i = 0, 1, ...) uses stage i % n at
// phase i / n. After `fills` fills were issued, wait (bounded) until the last
// fill of every stage has landed. A producer that leaves its loop early (a
// wait of its own or of another role gave up) calls this before the CTA
// exits, so that no copy it issued still writes the CTA's shared memory
// afterwards. Earlier fills of a stage have always landed (the next fill of a
// stage is issued only after its consumers released the previous one), so the
// parity wait cannot be satisfied by an older phase. Stages whose last fill
// was already consumed return at once.
__device__ __forceinline__ void drain_ring(uint64_t* full, int n_stages, uint32_t fills, uint32_t* status) {
    for (int s = 0; s < n_stages; ++s) {
        if (fills > (uint32_t)s) {
            const uint32_t last_use = (fills - 1 - (uint32_t)s) / (uint32_t)n_stages;
            mbar_wait_bounded(&full[s], last_use & 1u, status);
        }
    }
}

// Grid-wide barrier for a kernel whose CTAs are all resident (cooperative
// launch). count/gen live in global memory; count is 0 between barriers (the
// last arriver resets it before releasing the others). Arrival is a release
// (publishes the CTA's earlier writes, ordered by the preceding
// __syncthreads), the wait an acquire. Spins are bounded: on timeout the
// status word gets kStatusTimeout and false is returned.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Grid barrier on a monotonically increasing 64-bit arrival counter, for a
// kernel whose CTAs are all resident (cooperative launch). Every CTA adds 1
// (a release, publishing the CTA's writes ordered by the __syncthreads) and
// waits (acquire) until the counter reaches `target`, the base read at kernel
// start plus n_ctas per barrier passed. The counter is a multiple of n_ctas
// between kernels. Spins are bounded: on timeout the status word gets
// kStatusTimeout and false is returned.
struct GridSync {
    unsigned long long* count;
    unsigned long long base;
    uint32_t n;
    uint32_t passed;
};

// Call by every thread at kernel start, before this CTA's first arrival.
__device__ __forceinline__ GridSync grid_sync_init(unsigned long long* count, uint32_t n_ctas) {
    __shared__ unsigned long long s_base;
    if (threadIdx.x == 0) {
        const unsigned long long c = ld_acquire_gpu_u64(count);
        s_base = c - c % n_ctas;   // fewer than n_ctas arrivals can precede ours
    }
    __syncthreads();
    return GridSync{count, s_base, n_ctas, 0u};
}

// Split barrier: grid_arrive publishes this CTA's writes and counts it in;
// grid_wait (later, after independent work) waits for all CTAs of the same
// pass. grid_sync = grid_arrive + grid_wait.
__device__ __forceinline__ void grid_arrive(GridSync& gs) {
    __syncthreads();
    gs.passed += 1;
    if (threadIdx.x == 0) red_release_gpu_add_u64(gs.count, 1ull);
}

constexpr uint32_t kGridSpinLimit = 1u << 26;

__device__ __forceinline__ bool grid_wait(GridSync& gs, uint32_t* status, uint32_t limit = kGridSpinLimit) {
    __shared__ uint32_t s_okw;
    if (threadIdx.x == 0) {
        uint32_t ok = 1;
        const unsigned long long target = gs.base + (unsigned long long)gs.n * gs.passed;
        uint32_t it = 0;
        while (ld_acquire_gpu_u64(gs.count) < target) {
            if (++it > limit) {
                atomicOr(status, kStatusTimeout);
                ok = 0;
                break;
            }
            if (it > 256) __nanosleep(32);
        }
        s_okw = ok;
    }
    __syncthreads();
    return s_okw != 0;
}

__device__ __forceinline__ bool grid_sync(GridSync& gs, uint32_t* status) {
    __shared__ uint32_t s_ok;
    __syncthreads();
    gs.passed += 1;
    if (threadIdx.x == 0) {
        uint32_t ok = 1;
        const unsigned long long target = gs.base + (unsigned long long)gs.n * gs.passed;
        red_release_gpu_add_u64(gs.count, 1ull);
        uint32_t it = 0;
        while (ld_acquire_gpu_u64(gs.count) < target) {
            if (++it > kGridSpinLimit) {
                atomicOr(status, kStatusTimeout);
                ok = 0;
                break;
            }
            if (it > 256) __nanosleep(32);
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Grid barrier with the arrivals spread over kGridGroups counters, 128 bytes
// apart: CTA b counts into counter b % kGridGroups, so at most
// ceil(n_ctas / kGridGroups) same-address atomics queue at one L2 slice per
// barrier instead of n_ctas. A waiter polls all counters. Each counter is a
// multiple of its group's size between kernels. Same bounded waits as GridSync.
constexpr int kGridGroups = 8;
constexpr int kGridGroupStride = 16;   // unsigned long long: 128 bytes

struct GridSync8 {
    unsigned long long* count;   // [kGridGroups * kGridGroupStride]
    unsigned long long base[kGridGroups];
    uint32_t n_ctas;
    uint32_t passed;
};

__device__ __forceinline__ uint32_t grid_group_size(uint32_t n_ctas, int i) {
    return (n_ctas + kGridGroups - 1 - (uint32_t)i) / kGridGroups;
}

// Call by every thread at kernel start, before this CTA's first arrival.
__device__ __forceinline__ GridSync8 grid_sync8_init(unsigned long long* count, uint32_t n_ctas) {
    __shared__ unsigned long long s_base8[kGridGroups];
    if (threadIdx.x < kGridGroups) {
        const uint32_t n = grid_group_size(n_ctas, threadIdx.x);
        const unsigned long long c = ld_acquire_gpu_u64(count + threadIdx.x * kGridGroupStride);
        s_base8[threadIdx.x] = n ? c - c % n : c;   // fewer than n arrivals of this group can precede ours
    }
    __syncthreads();
    GridSync8 g;
    g.count = count;
#pragma unroll
    for (int i = 0; i < kGridGroups; ++i) g.base[i] = s_base8[i];
    g.n_ctas = n_ctas;
    g.passed = 0;
    return g;
}

// Split form: grid_arrive8 publishes this CTA's writes (ordered by its
// __syncthreads) and counts it in; grid_wait8, after independent work, waits
// for every CTA of the same pass. grid_sync8 = both.
__device__ __forceinline__ void grid_arrive8(GridSync8& gs) {
    __syncthreads();
    gs.passed += 1;
    if (threadIdx.x == 0) red_release_gpu_add_u64(gs.count + (blockIdx.x % kGridGroups) * kGridGroupStride, 1ull);
}

__device__ __forceinline__ bool grid_wait8(GridSync8& gs, uint32_t* status) {
    __shared__ uint32_t s_ok8;
    if (threadIdx.x == 0) {
        uint32_t ok = 1, it = 0;
        for (;;) {
            bool done = true;
            // relaxed polls (all eight in flight at once), then one fence:
            // the fence after observing every release makes this an acquire
#pragma unroll
            for (int i = 0; i < kGridGroups; ++i) {
                const unsigned long long target =
                    gs.base[i] + (unsigned long long)grid_group_size(gs.n_ctas, i) * gs.passed;
                const bool r = ld_relaxed_gpu_u64(gs.count + i * kGridGroupStride) >= target;
                done = done & r;
            }
            if (done) {
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                break;
            }
            if (++it > kGridSpinLimit) {
                atomicOr(status, kStatusTimeout);
                ok = 0;
                break;
            }
            if (it > 256) __nanosleep(32);
        }
        s_ok8 = ok;
    }
    __syncthreads();
    return s_ok8 != 0;
}

__device__ __forceinline__ bool grid_sync8(GridSync8& gs, uint32_t* status) {
    grid_arrive8(gs);
    return grid_wait8(gs, status);
}

}  // namespace flint
