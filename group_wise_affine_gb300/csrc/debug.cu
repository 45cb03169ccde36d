// Test exports: the unpacked integer codes and the fp32 dequantized weights,
// element by element, so the code layout and the dequantization step can be
// compared bit for bit with the CPU reference.  Formula: w = scale*q + bias
// ("saragossa", "Quantization formats": MLX affine integer weights), rounded
// once to fp32 by a fused multiply-add.
#include "common.cuh"
#include "internal.h"

namespace gwa {

// Code k of a row: bits [b*k, b*k + b) of the row's little-endian bit
// stream (a u3 or u6 code may take the top bits of one word and the bottom
// bits of the next; the next word is read only then).
__device__ __forceinline__ uint32_t row_code(const uint32_t *row, int64_t k,
                                             int bits) {
    const int64_t pos = (int64_t)bits * k;
    const int sh = (int)(pos & 31);
    const uint32_t lo = row[pos >> 5];
    const uint32_t v = sh + bits <= 32 ? lo >> sh
                                       : __funnelshift_r(lo, row[(pos >> 5) + 1], sh);
    return v & ((1u << bits) - 1u);
}

// One thread per code.
__global__ void debug_unpack_kernel(const uint32_t *__restrict__ wq, int64_t N,
                                    int64_t K, int bits,
                                    uint8_t *__restrict__ codes) {
    const int64_t wpr = K * bits / 32;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N * K;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / K, k = i - n * K;
        codes[i] = (uint8_t)row_code(wq + n * wpr, k, bits);
    }
}

__global__ void debug_dequant_kernel(const uint32_t *__restrict__ wq,
                                     const uint16_t *__restrict__ sc,
                                     const uint16_t *__restrict__ bi, int64_t N,
                                     int64_t K, int group, int bits,
                                     float *__restrict__ wf) {
    const int64_t wpr = K * bits / 32, G = K / group;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N * K;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / K, k = i - n * K;
        const float s = bf16_bits_to_f32(sc[n * G + k / group]);
        const float b = bf16_bits_to_f32(bi[n * G + k / group]);
        wf[i] = fmaf(s, (float)row_code(wq + n * wpr, k, bits), b);
    }
}

static unsigned grid_for(int64_t n, int threads) {
    int64_t g = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (g > cap) g = cap;
    return (unsigned)(g < 1 ? 1 : g);
}

cudaError_t launch_debug_unpack(const uint32_t *wq, int64_t N, int64_t K,
                                int bits, uint8_t *codes, cudaStream_t st) {
    debug_unpack_kernel<<<grid_for(N * K, 256), 256, 0, st>>>(wq, N, K, bits,
                                                              codes);
    return cudaGetLastError();
}

cudaError_t launch_debug_dequant(const uint32_t *wq, const uint16_t *sc,
                                 const uint16_t *bi, int64_t N, int64_t K,
                                 int bits, int group, float *wf,
                                 cudaStream_t st) {
    debug_dequant_kernel<<<grid_for(N * K, 256), 256, 0, st>>>(wq, sc, bi, N, K,
                                                               group, bits, wf);
    return cudaGetLastError();
}

}  // namespace gwa
