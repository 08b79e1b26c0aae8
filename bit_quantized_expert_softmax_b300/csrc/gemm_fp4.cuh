// Persistent block-scaled FP4 GEMM on the 5th-generation tensor cores
// (tcgen05.mma kind::mxf4nvf4, scale_vec::4X): D[128 x 128] (fp32, TMEM)
// += A[128 x K] . B[128 x K]^T with A and B packed E2M1 and one UE4M3 scale
// per 16 elements along K.
//
// Operands are stored in global memory already in the shared-memory image the
// MMA reads: a "block" (18 KiB) is one tile of 128 rows x 256 K-elements
// (16 KiB: 128 bytes per row, rows 128 bytes apart, the 16-byte chunk c of row
// r stored at chunk c ^ (r % 8), the 128-byte swizzle) followed by its scale
// factors (2 KiB: 128 rows x 16 bytes, row-major). The blocks of one row tile
// are contiguous along K, so one 1-D bulk copy moves two k-tiles of an operand,
// codes and scales, into shared memory: a stage is two copies of 36 KiB. (The
// bulk-copy engine moves ~0.3 us worth of copies at a time per SM whatever
// their size, so few large copies matter more than their count of bytes.)
//
// Warp roles of a CTA (448 threads, one CTA per SM):
//   warp 0      producer: bulk-copies A and B (two k-tiles each, with their
//               scales) into a ring of P::kStages stages
//   warp 1      allocates tensor memory; one thread issues the MMAs
//               (M=128, N=128, K=64 each; 4 per k-tile) into one of two
//               accumulators
//   warps 2..5  scale writers: shared memory -> tensor memory (tcgen05.st),
//               one row (lane) per thread
//   warps 6..13 epilogue: tensor memory -> registers -> the problem's store;
//               two warps per lane quadrant, each taking half of the 128
//               accumulator columns
// Tensor memory columns: accumulators [0,128) and [128,256); per stage s and
// k-tile i of the stage the A scales at 256+64s+32i..+15 and the B scales at
// 256+64s+32i+16..+31 (s < 4).
//
// Scale layout in tensor memory (per MMA of K = 64, 4 columns): lane m0 of
// every 32-lane quadrant, column m1 (0..3) holds the four UE4M3 scales (one
// per 16 K-elements, lowest K first) of tile row m0 + 32*m1; the four lane
// quadrants hold the same data. The MMA is given the first of its 4 columns.
#pragma once

#include "pdl.cuh"
#include "umma.cuh"

namespace flint {

constexpr int kGM = 128, kGN = 128, kGK = 256;
constexpr int kGTile = kGM * kGK / 2;          // 16 KiB of packed E2M1
constexpr int kGSf = kGM * kGK / 16;           // 2 KiB of UE4M3 scales
constexpr int kGBlk = kGTile + kGSf;           // one k-tile of one operand with its scales
constexpr int kGMaxStages = 4;                 // tensor-memory columns: 256 + 64 per stage
constexpr int kGThreads = 448;
constexpr int kGEpiWarps = 8;

// One output tile (or, with P::kNB = 2, a pair of output tiles sharing A) of
// a problem.
struct Fp4Item {
    const uint8_t* a;    // first block of A's row tile (blocks contiguous along K)
    const uint8_t* b;    // first block of B's row tile
    const uint8_t* b2;   // with kNB = 2: first block of the second B row tile
    int kt;              // number of k-tiles
    int m, n, aux;       // problem-defined (row tile, column tile, group)
};

// Layout of the engine for a problem with nb B tiles per item (1 or 2):
//   nb = 1: stage = [A blocks][B blocks]; two 128-column accumulators (the
//           epilogue of one item overlaps the MMAs of the next); per stage
//           64 scale-factor columns at 256 + 64s.
//   nb = 2: stage = [A blocks][B0 blocks][B1 blocks]; one accumulator pair
//           (256 columns: B0's tile, then B1's), single-buffered; per stage 96
//           scale-factor columns at 256 + 96s. Each A k-tile then feeds two
//           N-tiles: 3 blocks taken in per 2 block products instead of 4.
// (kps: k-tiles per stage, P::kKPS). With P::kBPair (kNB = 2 only) the two
// B row tiles of an item are stored interleaved by k-tile in global memory
// (B0 k-tile 0, B1 k-tile 0, B0 k-tile 1, ...), so one bulk copy brings both:
// two copies per stage instead of three (the bulk-copy engine's throughput
// per SM follows the number of copies in flight more than their size).
__host__ __device__ constexpr int fp4_stage_bytes(int nb, int kps) { return (1 + nb) * kps * kGBlk; }
__host__ __device__ constexpr int fp4_sf_cols(int nb, int kps) { return 16 * (1 + nb) * kps; }   // per stage

// Byte offset of element pair byte `j` (0..127) of row `r` (0..127) inside a
// swizzled tile.
__host__ __device__ __forceinline__ int swz_offset(int r, int j) {
    return r * 128 + ((((j >> 4) ^ (r & 7)) & 7) << 4) + (j & 15);
}

// Dynamic shared memory of the kernel for problem P (1024 bytes of slack for
// the 1024-byte alignment of the stage ring).
template <class P>
constexpr int fp4_gemm_smem() {
    static_assert(P::kStages >= 2 && P::kStages <= kGMaxStages, "stage count");
    static_assert(P::kNB == 1 || P::kNB == 2, "B tiles per item");
    static_assert(P::kKPS == 1 || P::kKPS == 2, "k-tiles per stage");
    static_assert(256 + fp4_sf_cols(P::kNB, P::kKPS) * P::kStages <= 512, "tensor-memory columns");
    return P::kStages * fp4_stage_bytes(P::kNB, P::kKPS) + kGEpiWarps * P::kEpiSmemPerWarp + 1024;
}

// A problem P provides kStages, kEpiSmemPerWarp, n_items(), item(i, w), a
// per-thread prologue pre(w, row, half) -> P::Pre (its loads are issued one
// item ahead, while the previous accumulator is being stored), the epilogue
// epilogue(w, pre, taddr, row, half, epi) of one accumulator (row = tile row
// of this thread, half = which 64 of the 128 columns, epi = kEpiSmemPerWarp
// bytes of shared memory owned by the warp) and epilogue_finish(), run once
// by every epilogue thread after its last item. Every role fetches the
// description of its next item before it waits on the current one.
template <class P>
__global__ void __launch_bounds__(kGThreads, 1) fp4_gemm_kernel(const P prob, uint32_t* status) {
    griddep_wait();
    extern __shared__ uint8_t graw[];
    constexpr int kGStages = P::kStages;
    constexpr int kNB = P::kNB;
    constexpr int kKPS = P::kKPS;
    constexpr int kStageB = fp4_stage_bytes(kNB, kKPS);
    constexpr int kSfCols = fp4_sf_cols(kNB, kKPS);
    constexpr bool kBPair = P::kBPair;
    static_assert(!kBPair || kNB == 2, "interleaved B needs two B tiles");
    // block index inside a stage of B tile b, k-tile i (A k-tile i is block i)
    auto bblk = [](int b, int i) { return kBPair ? kKPS + 2 * i + b : (1 + b) * kKPS + i; };
    constexpr int kNBuf = kNB == 1 ? 2 : 1;   // accumulator buffers
    __shared__ __align__(8) uint64_t full[kGStages], sfready[kGStages], empty[kGStages], accfull[2], accempty[2],
        mma_done;
    __shared__ uint32_t tmem_base;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(graw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&sfready[s], 4);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], kGEpiWarps);
        }
        mbar_init(&mma_done, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const int n_items = prob.n_items();

    if (warp == 0) {
        if (lane == 0) {
            uint32_t kcount = 0;
            bool ok = true;
            Fp4Item nxt;
            if ((int)blockIdx.x < n_items) prob.item(blockIdx.x, nxt);
            for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
                const Fp4Item w = nxt;
                if (i + (int)gridDim.x < n_items) prob.item(i + gridDim.x, nxt);
                for (int k0 = 0; k0 < w.kt; k0 += kKPS, ++kcount) {
                    const int s = kcount % kGStages;
                    const uint32_t use = kcount / kGStages;
                    if (use > 0 && !mbar_wait_bounded(&empty[s], (use - 1) & 1, status)) {
                        ok = false;
                        break;
                    }
                    const int n = w.kt - k0 < kKPS ? w.kt - k0 : kKPS;
                    uint8_t* st = sm + s * kStageB;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)((1 + kNB) * n * kGBlk));
                    bulk_g2s(st, w.a + (size_t)k0 * kGBlk, (uint32_t)(n * kGBlk), &full[s]);
                    if constexpr (kBPair) {
                        bulk_g2s(st + kKPS * kGBlk, w.b + (size_t)2 * k0 * kGBlk, (uint32_t)(2 * n * kGBlk), &full[s]);
                    } else {
                        bulk_g2s(st + kKPS * kGBlk, w.b + (size_t)k0 * kGBlk, (uint32_t)(n * kGBlk), &full[s]);
                        if constexpr (kNB == 2)
                            bulk_g2s(st + 2 * kKPS * kGBlk, w.b2 + (size_t)k0 * kGBlk, (uint32_t)(n * kGBlk),
                                     &full[s]);
                    }
                }
            }
            // every copy issued has landed before the CTA can exit, also when
            // a role gave up early
            drain_ring(full, kGStages, kcount, status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_nvfp4_f32(kGM, kGN);
            uint32_t kcount = 0, n_done = 0;
            bool ok = true;
            Fp4Item nxt;
            if ((int)blockIdx.x < n_items) prob.item(blockIdx.x, nxt);
            for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
                const Fp4Item w = nxt;
                if (i + (int)gridDim.x < n_items) prob.item(i + gridDim.x, nxt);
                const uint32_t buf = n_done % kNBuf;
                if (n_done >= (uint32_t)kNBuf &&
                    !mbar_wait_bounded(&accempty[buf], ((n_done / kNBuf) - 1) & 1, status))
                    break;
                tc_fence_after();
                const uint32_t acc = tmem + buf * kGN;
                for (int k0 = 0; k0 < w.kt; k0 += kKPS, ++kcount) {
                    const int s = kcount % kGStages;
                    const uint32_t use = kcount / kGStages;
                    if (!mbar_wait_bounded(&sfready[s], use & 1, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int n = w.kt - k0 < kKPS ? w.kt - k0 : kKPS;
                    const uint8_t* st = sm + s * kStageB;
                    for (int i = 0; i < n; ++i) {
                        const uint64_t da = sdesc_kmajor_sw128(st + i * kGBlk);
                        // scale columns of k-tile i: A at +0, B0 at +16, B1 at +32
                        const uint32_t sfa = tmem + 256 + kSfCols * s + 16 * (1 + kNB) * i;
#pragma unroll
                        for (int b = 0; b < kNB; ++b) {
                            const uint64_t db = sdesc_kmajor_sw128(st + bblk(b, i) * kGBlk);
                            const uint32_t sfb = sfa + 16 * (1 + b);
#pragma unroll
                            for (int j = 0; j < 4; ++j)   // 64 E2M1 = 32 bytes = 2 descriptor units per MMA
                                umma_nvfp4(acc + b * kGN, da + 2 * j, db + 2 * j, idesc, sfa + 4 * j, sfb + 4 * j,
                                           (k0 | i | j) != 0);
                        }
                    }
                    umma_commit(&empty[s]);
                }
                umma_commit(&accfull[buf]);
                ++n_done;
            }
            // every MMA issued has completed before the tensor memory is
            // released, also when a wait gave up early
            umma_commit(&mma_done);
            mbar_wait_bounded(&mma_done, 0, status);
        }
    } else if (warp < 6) {
        // scale writers: every quadrant writes the same 32 x 16-byte image:
        // thread (quadrant, lane m0) stores rows m0, m0+32, m0+64, m0+96
        const int quad = warp & 3;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint32_t kcount = 0;
        bool ok = true;
        Fp4Item nxt;
        if ((int)blockIdx.x < n_items) prob.item(blockIdx.x, nxt);
        for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
            const Fp4Item w = nxt;
            if (i + (int)gridDim.x < n_items) prob.item(i + gridDim.x, nxt);
            for (int k0 = 0; k0 < w.kt; k0 += kKPS, ++kcount) {
                const int s = kcount % kGStages;
                const uint32_t use = kcount / kGStages;
                const bool got = mbar_wait_bounded(&full[s], use & 1, status);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const int n = w.kt - k0 < kKPS ? w.kt - k0 : kKPS;
                const uint8_t* st = sm + s * kStageB;
                for (int q = 0; q < (1 + kNB) * n; ++q) {
                    const int i = q / (1 + kNB), op = q % (1 + kNB);   // op 0: A, 1 + b: B tile b
                    const uint8_t* sf = st + (op == 0 ? i : bblk(op - 1, i)) * kGBlk + kGTile;
                    uint4 r[4];
#pragma unroll
                    for (int m1 = 0; m1 < 4; ++m1) r[m1] = *reinterpret_cast<const uint4*>(sf + (lane + 32 * m1) * 16);
                    const uint32_t col = tmem + lane_base + 256 + kSfCols * s + 16 * (1 + kNB) * i + 16 * op;
                    // MMA j (K elements 64j..64j+63) reads word j of each row
                    tmem_st4(col + 0, r[0].x, r[1].x, r[2].x, r[3].x);
                    tmem_st4(col + 4, r[0].y, r[1].y, r[2].y, r[3].y);
                    tmem_st4(col + 8, r[0].z, r[1].z, r[2].z, r[3].z);
                    tmem_st4(col + 12, r[0].w, r[1].w, r[2].w, r[3].w);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfready[s]);
            }
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31 and the
        // columns [64*half, 64*half + 64) of the accumulator
        const int quad = warp & 3;
        const int half = (warp - 6) >> 2;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint8_t* epi = sm + kGStages * kStageB + (warp - 6) * P::kEpiSmemPerWarp;
        uint32_t n_done = 0;
        Fp4Item nxt;
        typename P::Pre pnxt{};
        if ((int)blockIdx.x < n_items) {
            prob.item(blockIdx.x, nxt);
            pnxt = prob.pre(nxt, row, half);
        }
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            const Fp4Item w = nxt;
            const typename P::Pre pw = pnxt;
            if (i + (int)gridDim.x < n_items) {
                prob.item(i + gridDim.x, nxt);
                pnxt = prob.pre(nxt, row, half);
            }
            const uint32_t buf = n_done % kNBuf;
            const bool got = mbar_wait_bounded(&accfull[buf], (n_done / kNBuf) & 1, status);
            // all epilogue warps agree on the outcome (named barrier 2), so a
            // problem's epilogue may synchronise them (named barrier 1)
            // without waiting for a warp that has left
            uint32_t all_got;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\t"
                "setp.ne.u32 p, %1, 0;\n\t"
                "barrier.cta.red.and.pred q, 2, %2, p;\n\t"
                "selp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(all_got)
                : "r"((uint32_t)got), "n"(kGEpiWarps * 32)
                : "memory");
            if (!all_got) break;
            tc_fence_after();
            // the problem's epilogue reads the accumulator(s) and calls
            // release() as soon as it no longer needs tensor memory
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&accempty[buf]);
            };
            prob.epilogue(w, pw, tmem + lane_base + buf * kGN, row, half, epi, release);
            ++n_done;
        }
        prob.epilogue_finish();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace flint

namespace flint {

// ---------------------------------------------------------------------------
// Variant with a resident A operand, for products whose K is short (two
// k-tiles): a work item is one 128-row A tile (an "M-tile") and all P::kNT
// B tiles of its expert. The A tile (codes and scales of its kKT k-tiles) is
// bulk-copied once into one of two A slots and its scale factors written to
// tensor memory once; the B tiles stream through a ring of P::kStages stages
// of one N-tile each (kKT k-tiles), and each N-tile's accumulator goes to the
// epilogue as in fp4_gemm_kernel. Per M-tile the SMs take in one A tile plus
// the expert's B tiles instead of one A tile per N-tile.
//
// Roles: warp 0 producer (A tiles one M-tile ahead, B tiles); warp 1 tensor
// memory and MMA issue; warps 2..5 scale writers (A scales once per M-tile,
// B scales per stage); warps 6..13 epilogue. Tensor memory: accumulators
// [0,256), A scales of slot a at 256 + 32a (k-tile i: + 16i), B scales of
// stage s at 320 + 32s (k-tile i: + 16i).
// ---------------------------------------------------------------------------
constexpr int kRKT = 2;                        // k-tiles per item (K = 512)
constexpr int kRStageBytes = kRKT * kGBlk;     // one N-tile of B, or one A tile

template <class P>
constexpr int fp4_gemm_resa_smem() {
    static_assert(P::kStages >= 2 && 320 + 32 * P::kStages <= 512, "tensor-memory columns");
    return 2 * kRStageBytes + P::kStages * kRStageBytes + kGEpiWarps * P::kEpiSmemPerWarp + 1024;
}

template <class P>
__global__ void __launch_bounds__(kGThreads, 1) fp4_gemm_resa_kernel(const P prob, uint32_t* status) {
    griddep_wait();
    extern __shared__ uint8_t graw[];
    constexpr int kS = P::kStages;
    constexpr int kNT = P::kNT;
    __shared__ __align__(8) uint64_t full[kS], sfready[kS], empty[kS], afull[2], asfready[2], aempty[2],
        accfull[2], accempty[2], mma_done;
    __shared__ uint32_t tmem_base;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(graw) + 1023) & ~uintptr_t(1023));
    uint8_t* aslot = sm;                                  // [2][kRStageBytes]
    uint8_t* bring = sm + 2 * kRStageBytes;               // [kS][kRStageBytes]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&sfready[s], 4);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&afull[b], 1);
            mbar_init(&asfready[b], 4);
            mbar_init(&aempty[b], 1);
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], kGEpiWarps);
        }
        mbar_init(&mma_done, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const int n_mt = prob.n_mtiles();

    if (warp == 0) {
        if (lane == 0) {
            uint32_t bfills = 0, afills = 0;
            bool ok = true;
            for (int mt = blockIdx.x; mt < n_mt && ok; mt += gridDim.x, ++afills) {
                const int a = afills & 1;
                if (afills >= 2 && !mbar_wait_bounded(&aempty[a], ((afills >> 1) - 1) & 1, status)) break;
                mbar_arrive_expect_tx(&afull[a], kRStageBytes);
                bulk_g2s(aslot + a * kRStageBytes, prob.a_blocks(mt), kRStageBytes, &afull[a]);
                for (int n = 0; n < kNT; ++n, ++bfills) {
                    const int s = bfills % kS;
                    const uint32_t use = bfills / kS;
                    if (use > 0 && !mbar_wait_bounded(&empty[s], (use - 1) & 1, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], kRStageBytes);
                    bulk_g2s(bring + s * kRStageBytes, prob.b_blocks(mt, n), kRStageBytes, &full[s]);
                }
            }
            // every copy issued has landed before the CTA can exit
            drain_ring(full, kS, bfills, status);
            drain_ring(afull, 2, afills, status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_nvfp4_f32(kGM, kGN);
            uint32_t bcount = 0, n_done = 0, acount = 0;
            bool ok = true;
            for (int mt = blockIdx.x; mt < n_mt && ok; mt += gridDim.x, ++acount) {
                const int a = acount & 1;
                if (!mbar_wait_bounded(&asfready[a], (acount >> 1) & 1, status)) break;
                tc_fence_after();
                for (int n = 0; n < kNT; ++n, ++bcount) {
                    const uint32_t buf = n_done & 1;
                    if (n_done >= 2 && !mbar_wait_bounded(&accempty[buf], ((n_done >> 1) - 1) & 1, status)) {
                        ok = false;
                        break;
                    }
                    const int s = bcount % kS;
                    if (!mbar_wait_bounded(&sfready[s], (bcount / kS) & 1, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc = tmem + buf * kGN;
                    for (int i = 0; i < kRKT; ++i) {
                        const uint64_t da = sdesc_kmajor_sw128(aslot + a * kRStageBytes + i * kGBlk);
                        const uint64_t db = sdesc_kmajor_sw128(bring + s * kRStageBytes + i * kGBlk);
                        const uint32_t sfa = tmem + 256 + 32 * a + 16 * i, sfb = tmem + 320 + 32 * s + 16 * i;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            umma_nvfp4(acc, da + 2 * j, db + 2 * j, idesc, sfa + 4 * j, sfb + 4 * j, (i | j) != 0);
                    }
                    umma_commit(&empty[s]);
                    umma_commit(&accfull[buf]);
                    ++n_done;
                }
                umma_commit(&aempty[a]);   // the A slot and its scale columns are free once these MMAs finish
            }
            umma_commit(&mma_done);
            mbar_wait_bounded(&mma_done, 0, status);
        }
    } else if (warp < 6) {
        // scale writers: every quadrant writes the same 32 x 16-byte image
        const int quad = warp & 3;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        auto write_sf = [&](const uint8_t* blk_scales, uint32_t col) {
            uint4 r[4];
#pragma unroll
            for (int m1 = 0; m1 < 4; ++m1) r[m1] = *reinterpret_cast<const uint4*>(blk_scales + (lane + 32 * m1) * 16);
            tmem_st4(col + 0, r[0].x, r[1].x, r[2].x, r[3].x);
            tmem_st4(col + 4, r[0].y, r[1].y, r[2].y, r[3].y);
            tmem_st4(col + 8, r[0].z, r[1].z, r[2].z, r[3].z);
            tmem_st4(col + 12, r[0].w, r[1].w, r[2].w, r[3].w);
        };
        uint32_t bcount = 0, acount = 0;
        bool ok = true;
        for (int mt = blockIdx.x; mt < n_mt && ok; mt += gridDim.x, ++acount) {
            const int a = acount & 1;
            const bool got = mbar_wait_bounded(&afull[a], (acount >> 1) & 1, status);
            if (!__all_sync(0xffffffffu, got)) break;
            for (int i = 0; i < kRKT; ++i)
                write_sf(aslot + a * kRStageBytes + i * kGBlk + kGTile, tmem + lane_base + 256 + 32 * a + 16 * i);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&asfready[a]);
            for (int n = 0; n < kNT; ++n, ++bcount) {
                const int s = bcount % kS;
                const bool gotb = mbar_wait_bounded(&full[s], (bcount / kS) & 1, status);
                if (!__all_sync(0xffffffffu, gotb)) {
                    ok = false;
                    break;
                }
                for (int i = 0; i < kRKT; ++i)
                    write_sf(bring + s * kRStageBytes + i * kGBlk + kGTile, tmem + lane_base + 320 + 32 * s + 16 * i);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfready[s]);
            }
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31 and the
        // columns [64*half, 64*half + 64) of the accumulator
        const int quad = warp & 3;
        const int half = (warp - 6) >> 2;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint8_t* epi = sm + 2 * kRStageBytes + kS * kRStageBytes + (warp - 6) * P::kEpiSmemPerWarp;
        uint32_t n_done = 0;
        bool ok = true;
        for (int mt = blockIdx.x; mt < n_mt && ok; mt += gridDim.x) {
            const typename P::Pre pw = prob.pre(mt, row, half);
            for (int n = 0; n < kNT; ++n) {
                const uint32_t buf = n_done & 1;
                const bool got = mbar_wait_bounded(&accfull[buf], (n_done >> 1) & 1, status);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                prob.epilogue(mt, n, pw, tmem + lane_base + buf * kGN, row, half, epi);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&accempty[buf]);
                ++n_done;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace flint
