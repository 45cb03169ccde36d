// Test exports: the unpacked integer codes and the fp32 dequantized weights,
// element by element, so the code layout and the dequantization step can be
// compared bit for bit with the CPU reference.  Formula: w = scale*q + bias
// ("saragossa", "Quantization formats": MLX affine integer weights; fp8
// codes stand for their E4M3 numbers), rounded once to fp32 by a fused
// multiply-add.
#include "common.cuh"
#include "internal.h"

namespace gwa {

// Code k of a row: bits [b*k, b*k + b) of the row's little-endian bit
// stream (a u3 or u6 code may take the top bits of one word and the bottom
// bits of the next; the next word is read only then).
__device__ __forceinline__ uint32_t row_code(const uint32_t *row, int64_t k,
                                             int bits) {
    bits = code_bits(bits);
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
    const int64_t wpr = K * code_bits(bits) / 32;
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
    const int64_t wpr = K * code_bits(bits) / 32, G = K / group;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N * K;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / K, k = i - n * K;
        const float s = bf16_bits_to_f32(sc[n * G + k / group]);
        const float b = bf16_bits_to_f32(bi[n * G + k / group]);
        const uint32_t c = row_code(wq + n * wpr, k, bits);
        wf[i] = fmaf(s, bits == kFp8 ? e4m3_to_f32(c) : (float)c, b);
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

// The bounded pipeline wait, made to run out: one CTA, an mbarrier that
// expects one arrival which never comes.  Warp 0 waits with mbar_wait
// (the streaming and decode kernels' wait), warp 1 with mbar_wait_sleep
// (the tensor-core kernel's), both with `limit_ns` in place of the kernels'
// 2 s.  out[2w] = 1 when warp w's wait gave up (0 if it completed),
// out[2w + 1] = the microseconds it waited.  Nothing is left in flight: the
// barrier guards no copy, so the CTA can simply return.
__global__ void debug_wait_kernel(uint32_t *out, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int w = threadIdx.x / kWarp;
    const unsigned long long t0 = global_ns();
    const bool ok = w == 0 ? mbar_wait(&bar, 0, limit_ns)
                           : mbar_wait_sleep(&bar, 0, limit_ns);
    const unsigned long long t1 = global_ns();
    if ((threadIdx.x & (kWarp - 1)) == 0) {
        out[2 * w] = ok ? 0u : 1u;
        out[2 * w + 1] = (uint32_t)((t1 - t0) / 1000ull);
    }
}

cudaError_t launch_debug_wait(uint32_t *out, unsigned long long limit_ns,
                              cudaStream_t st) {
    debug_wait_kernel<<<1, 2 * kWarp, 0, st>>>(out, limit_ns);
    return cudaGetLastError();
}

}  // namespace gwa
