// Test exports: the unpacked integer codes and the fp32 dequantized weights,
// element by element, so the code layout and the dequantization step can be
// compared bit for bit with the CPU reference.  Formula: w = scale*q + bias
// ("saragossa", "Quantization formats": MLX affine integer weights), rounded
// once to fp32 by a fused multiply-add.
#include "common.cuh"
#include "internal.h"

namespace gwa {

__global__ void debug_unpack_kernel(const uint32_t *__restrict__ wq,
                                    int64_t words, int bits,
                                    uint8_t *__restrict__ codes) {
    const int per = 32 / bits;
    const uint32_t mask = (1u << bits) - 1u;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t w = wq[i];
        for (int j = 0; j < per; ++j)
            codes[i * per + j] = (uint8_t)((w >> (bits * j)) & mask);
    }
}

__global__ void debug_dequant_kernel(const uint32_t *__restrict__ wq,
                                     const uint16_t *__restrict__ sc,
                                     const uint16_t *__restrict__ bi,
                                     int64_t words, int64_t words_per_row,
                                     int64_t G, int group, int bits,
                                     float *__restrict__ wf) {
    const int per = 32 / bits;
    const uint32_t mask = (1u << bits) - 1u;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / words_per_row, wi = i - n * words_per_row;
        const uint32_t w = wq[i];
        for (int j = 0; j < per; ++j) {
            const int64_t k = wi * per + j;
            const float s = bf16_bits_to_f32(sc[n * G + k / group]);
            const float b = bf16_bits_to_f32(bi[n * G + k / group]);
            wf[i * per + j] = fmaf(s, (float)((w >> (bits * j)) & mask), b);
        }
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
    const int64_t words = N * K * bits / 32;
    debug_unpack_kernel<<<grid_for(words, 256), 256, 0, st>>>(wq, words, bits,
                                                              codes);
    return cudaGetLastError();
}

cudaError_t launch_debug_dequant(const uint32_t *wq, const uint16_t *sc,
                                 const uint16_t *bi, int64_t N, int64_t K,
                                 int bits, int group, float *wf,
                                 cudaStream_t st) {
    const int64_t words = N * K * bits / 32;
    debug_dequant_kernel<<<grid_for(words, 256), 256, 0, st>>>(
        wq, sc, bi, words, K * bits / 32, K / group, group, bits, wf);
    return cudaGetLastError();
}

}  // namespace gwa
