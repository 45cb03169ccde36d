// Decode kernel for the code widths and group sizes outside the tuned ones
// (u4/u8 at group 64): u2, u4, u8 codes with groups of 32, 64 or 128 inputs
// ("saragossa", "Quantization formats": MLX affine integer weights at
// several widths; the group size is a parameter of MLX's quantized_matmul).
// Same packed format: P = 32/b codes per word along the input axis, lowest
// bits first; one bf16 scale and bias per group; w = scale * q + bias.
//
// One warp per output unit (a row, or a gate/up or rotary pair of rows):
// the lanes stride over the row's 32-bit words (a word never spans two
// groups, since every group is a multiple of P codes), form each weight in
// fp32 and accumulate its products with up to four tokens, reading the
// activations straight from global memory (a few KB, cached in L1 and L2
// across all rows; a word's activations are one 8-32-byte read per token).
// A warp reduction and the same epilogues as the tuned kernels (plain,
// sections with bias, SiLU(gate) * up, rotary pairs) finish it.  It trades
// speed for generality: about four instructions per code and token.
#include "common.cuh"
#include "internal.h"

namespace gwa {

constexpr int kGenTokens = 4;   // tokens per pass
constexpr int kGenThreads = 256;

template <int BITS, int MODE>
__global__ void __launch_bounds__(kGenThreads)
    qmv_generic_kernel(DenseParams p, int64_t units) {
    constexpr int P = 32 / BITS;
    constexpr uint32_t MASK = (1u << BITS) - 1u;
    constexpr bool PAIRS = MODE == 2 || MODE == 3;
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / kWarp;
    const int64_t wpr = (int64_t)p.K / P;  // words per row
    const int64_t I = p.N / 2;
    const int gshift = __ffs(p.group) - 1;  // groups are 32, 64 or 128
    if (threadIdx.x == 0) pdl_launch_dependents();
    pdl_wait_primary();  // x may be the previous kernel's output
    for (int64_t u = warp; u < units; u += nwarps) {
        int64_t rows[2];
        if (MODE == 2) {
            rows[0] = u;
            rows[1] = I + u;
        } else if (MODE == 3) {
            rows[0] = rope_pair_row(u, 0, p.rope_hd);
            rows[1] = rope_pair_row(u, 1, p.rope_hd);
        } else {
            rows[0] = rows[1] = u;
        }
        float acc[2][kGenTokens];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int m = 0; m < kGenTokens; ++m) acc[h][m] = 0.f;
#pragma unroll
        for (int h = 0; h < (PAIRS ? 2 : 1); ++h) {
            const uint32_t *wrow = p.wq + rows[h] * wpr;
            const uint16_t *srow = p.sc + rows[h] * p.G;
            const uint16_t *brow = p.bi + rows[h] * p.G;
            // a lane takes words wi, wi + 32, wi + 64, wi + 96 per step: four
            // loads in flight, each a contiguous 128 bytes across the warp,
            // and the activations of consecutive lanes stay contiguous too
            // (rows are whole multiples of 128 words when K % 512 == 0;
            // shorter tails are masked)
            for (int64_t w0 = 0; w0 < wpr; w0 += 4 * kWarp) {
                uint32_t words[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int64_t wi = w0 + q4 * kWarp + lane;
                    words[q4] = wi < wpr ? wrow[wi] : 0u;
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int64_t wi = w0 + q4 * kWarp + lane;
                    if (wi >= wpr) break;
                    const int64_t k0 = wi * P;
                    const int g = (int)(k0 >> gshift);  // one group per word
                    const float s = bf16_bits_to_f32(srow[g]);
                    const float b = bf16_bits_to_f32(brow[g]);
                    float wv[P];
#pragma unroll
                    for (int c = 0; c < P; ++c) {
                        // the code as a float: 2^23 + q minus 2^23 (exact)
                        const float q = __uint_as_float(
                            0x4b000000u | ((words[q4] >> (BITS * c)) & MASK)) -
                                        8388608.0f;
                        wv[c] = fmaf(s, q, b);
                    }
#pragma unroll
                    for (int m = 0; m < kGenTokens; ++m) {
                        if (m >= p.M) break;
                        // the word's P activations of token m (2P bytes)
                        const uint32_t *xw = reinterpret_cast<const uint32_t *>(
                            p.x + (int64_t)m * p.K + k0);
#pragma unroll
                        for (int c2 = 0; c2 < P / 2; ++c2) {
                            const uint32_t pr = xw[c2];
                            acc[h][m] = fmaf(wv[2 * c2], bf16_lo(pr), acc[h][m]);
                            acc[h][m] = fmaf(wv[2 * c2 + 1], bf16_hi(pr), acc[h][m]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int m = 0; m < kGenTokens; ++m)
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
                    acc[h][m] += __shfl_xor_sync(0xffffffffu, acc[h][m], o);
        if (lane >= kGenTokens || lane >= p.M) continue;
        // lane m writes token m (a compile-time index below)
#pragma unroll
        for (int m = 0; m < kGenTokens; ++m) {
            if (m != lane) continue;
            if constexpr (MODE == 0) {
                p.y[(int64_t)m * p.N + u] = f32_to_bf16_bits(acc[0][m]);
            } else if constexpr (MODE == 2) {
                const float gv = acc[0][m], uv = acc[1][m];
                p.y[(int64_t)m * I + u] =
                    f32_to_bf16_bits(gv / (1.0f + __expf(-gv)) * uv);
            } else {
                const int64_t r0 = rows[0];
                int s = 0;
                while (s + 1 < p.nsec && r0 >= p.sec_start[s + 1]) ++s;
                const int64_t j = r0 - p.sec_start[s];
                const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
                float a = acc[0][m];
                if (p.sec_bias[s]) a += bf16_bits_to_f32(p.sec_bias[s][j]);
                if constexpr (MODE == 1) {
                    p.sec_out[s][(int64_t)m * size + j] = f32_to_bf16_bits(a);
                } else {
                    const int half = p.rope_hd / 2;
                    float c = acc[1][m];
                    if (p.sec_bias[s]) c += bf16_bits_to_f32(p.sec_bias[s][j + half]);
                    if (r0 < p.rope_end) {
                        const float2 t =
                            p.rope_cs[(int64_t)m * half + (int)(u % half)];
                        const float a2 = a * t.x - c * t.y;
                        c = c * t.x + a * t.y;
                        a = a2;
                    }
                    uint16_t *o = p.sec_out[s] + (int64_t)m * size + j;
                    o[0] = f32_to_bf16_bits(a);
                    o[half] = f32_to_bf16_bits(c);
                }
            }
        }
    }
}

template <int BITS>
static cudaError_t launch_generic_b(int mode, const DenseParams &p,
                                    cudaStream_t st) {
    const int64_t units = mode == 2 || mode == 3 ? p.N / 2 : p.N;
    if (units <= 0) return cudaSuccess;
    int64_t grid = (units + kGenThreads / kWarp - 1) / (kGenThreads / kWarp);
    const int64_t cap = (int64_t)num_sms() * (2048 / kGenThreads);
    if (grid > cap) grid = cap;
    const void *k = mode == 0   ? reinterpret_cast<const void *>(qmv_generic_kernel<BITS, 0>)
                    : mode == 1 ? reinterpret_cast<const void *>(qmv_generic_kernel<BITS, 1>)
                    : mode == 2 ? reinterpret_cast<const void *>(qmv_generic_kernel<BITS, 2>)
                                : reinterpret_cast<const void *>(qmv_generic_kernel<BITS, 3>);
    return launch_pdl(k, (unsigned)grid, (unsigned)kGenThreads, 0, st, p, units);
}

// Runs the general-format kernel over passes of up to kGenTokens tokens;
// `mode` as the other decode kernels (0 plain, 1 sections, 2 gate+up, 3
// sections with the rotary embedding from p.rope_cs).
cudaError_t launch_generic(int mode, const DenseParams &p, cudaStream_t st) {
    return p.bits == 2   ? launch_generic_b<2>(mode, p, st)
           : p.bits == 4 ? launch_generic_b<4>(mode, p, st)
                         : launch_generic_b<8>(mode, p, st);
}

int generic_max_tokens() { return kGenTokens; }

}  // namespace gwa
