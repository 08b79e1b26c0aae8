// Weight repacking (canonical row-major -> tiled mma-fragment layout) and the
// dequantisation export used to check the device layout bit for bit.
#include "kernels.cuh"
#include "tiles.cuh"

namespace flint {

namespace {

__global__ void repack_kernel(const uint8_t* __restrict__ codes_src, const uint8_t* __restrict__ scales_src,
                              uint8_t* __restrict__ codes_dst, uint8_t* __restrict__ scales_dst, int R,
                              int K, int wfmt) {
    const int KT = K >> 7;
    const long n_lanes = (long)(R >> 3) * KT * 32;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n_lanes; i += (long)gridDim.x * blockDim.x) {
        const int lane = (int)(i & 31);
        const long tile = i >> 5;
        const int kt = (int)(tile % KT), rt = (int)(tile / KT);
        const int g = lane >> 2, c = lane & 3;
        const int row = rt * 8 + g;
        const uint8_t* src = codes_src + (size_t)row * (K / 2) + kt * 64;
        uint8_t v[16];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            v[2 * s] = src[8 * s + c];
            v[2 * s + 1] = src[8 * s + c + 4];
        }
        uint4 o;
        o.x = v[0] | (v[1] << 8) | (v[2] << 16) | ((uint32_t)v[3] << 24);
        o.y = v[4] | (v[5] << 8) | (v[6] << 16) | ((uint32_t)v[7] << 24);
        o.z = v[8] | (v[9] << 8) | (v[10] << 16) | ((uint32_t)v[11] << 24);
        o.w = v[12] | (v[13] << 8) | (v[14] << 16) | ((uint32_t)v[15] << 24);
        *reinterpret_cast<uint4*>(codes_dst + tile * 512 + lane * 16) = o;
        if (c == 0) {
            if (wfmt == 0) {
                const uint8_t* ss = scales_src + (size_t)row * (K / 16) + kt * 8;
                uint8_t* sd = scales_dst + tile * 64 + g * 8;
#pragma unroll
                for (int s = 0; s < 8; ++s) sd[s] = ss[s];
            } else {
                const uint8_t* ss = scales_src + (size_t)row * (K / 32) * 4 + kt * 16;
                uint8_t* sd = scales_dst + tile * 128 + g * 16;
#pragma unroll
                for (int b = 0; b < 16; ++b) sd[b] = ss[b];
            }
        }
    }
}

// One thread per canonical element (row, k): locate its byte in the tiled
// layout and decode it with the decoders the expert kernels use (tiles.cuh):
// NVFP4 fp32(E2M1 x E4M3 x tensor scale), q4_1 fp32(d*q + m).
__global__ void dequant_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                               const float* __restrict__ tscale_dev, float tscale_host, int R, int K,
                               int wfmt, float* __restrict__ out) {
    const int KT = K >> 7;
    const long n = (long)R * K;
    const float ts = tscale_dev != nullptr ? *tscale_dev : tscale_host;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int row = (int)(i / K), k = (int)(i % K);
        const int rt = row >> 3, g = row & 7, kt = k >> 7, kk = k & 127;
        const int s = kk >> 4, r = kk & 15;
        const int c = (r & 7) >> 1;
        const int hi_half = r >> 3;        // 2c+8.. lives in the second byte of the step
        const int nib = r & 1;
        const long tile = (long)rt * KT + kt;
        const int lane = g * 4 + c;
        const uint8_t byte = codes[tile * 512 + lane * 16 + 2 * s + hi_half];
        float v;
        if (wfmt == 0) {
            v = nvfp4_code_times_scale(byte, nib, scales[tile * 64 + g * 8 + s]) * ts;
        } else {
            const uint32_t dm = *reinterpret_cast<const uint32_t*>(scales + tile * 128 + g * 16 + (s >> 1) * 4);
            v = q41_weight(byte, nib, dm);
        }
        out[i] = v;
    }
}

}  // namespace

cudaError_t launch_repack_matrix(const uint8_t* codes_src, const uint8_t* scales_src,
                                 uint8_t* codes_dst, uint8_t* scales_dst, int R, int K, int wfmt,
                                 cudaStream_t st) {
    const long n_lanes = (long)(R / 8) * (K / 128) * 32;
    long blocks = (n_lanes + 255) / 256;
    if (blocks > 148 * 16) blocks = 148 * 16;
    repack_kernel<<<(int)blocks, 256, 0, st>>>(codes_src, scales_src, codes_dst, scales_dst, R, K, wfmt);
    return cudaGetLastError();
}

cudaError_t launch_dequant_matrix(const uint8_t* codes, const uint8_t* scales, float tscale_host,
                                  const float* tscale_dev, int R, int K, int wfmt, float* out,
                                  cudaStream_t st) {
    const long n = (long)R * K;
    long blocks = (n + 255) / 256;
    if (blocks > 148 * 16) blocks = 148 * 16;
    dequant_kernel<<<(int)blocks, 256, 0, st>>>(codes, scales, tscale_dev, tscale_host, R, K, wfmt, out);
    return cudaGetLastError();
}

}  // namespace flint
