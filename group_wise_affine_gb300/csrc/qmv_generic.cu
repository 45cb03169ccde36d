// Decode kernel for the code widths and group sizes outside the tuned ones
// (u4/u8 at group 64): u2, u3, u4, u6, u8 codes with groups of 32, 64 or
// 128 inputs ("saragossa", "Quantization formats": MLX affine integer
// weights u2/u3/u4/u6/u8; the group size is a parameter of MLX's
// quantized_matmul).  Same packed format: a row's words are one
// little-endian bit stream, code k at bits [b*k, b*k + b), lowest bits
// first (field k mod 32/b of word k*b/32 for the widths that divide 32; a
// u3 or u6 code may straddle two words); one bf16 scale and bias per group;
// w = scale * q + bias.  fp8 (e4m3) codes in the same container (bits =
// GWA_FP8_E4M3, four bytes a word) take the fp32 kernel below with each
// code's E4M3 value in place of the integer: w = scale * e4m3(q) + bias.
//
// One warp per output unit (a row, or a gate/up or rotary pair of rows):
// the lanes stride over the row in code units -- one word (32/b codes) for
// the widths that divide 32, three words (96 bits: 32 u3 or 16 u6 codes)
// for the others -- so a unit never spans two groups and starts on a code
// boundary.  Each lane forms its unit's weights in fp32 (a straddling code
// by a funnel shift of two words) and accumulates their products with up to
// four tokens, reading the activations straight from global memory (a few
// KB, cached in L1 and L2 across all rows).  A warp reduction and the same
// epilogues as the tuned kernels (plain, sections with bias, SiLU(gate) *
// up, rotary pairs) finish it.  It trades speed for generality: about four
// instructions per code and token.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gwa {

constexpr int kGenTokens = 4;   // tokens per pass
constexpr int kGenThreads = 256;

// Words per code unit and codes per unit of a width (fp8: four words, 16
// codes, so that a lane's unit is one 16-byte load).
template <int BITS>
struct GenUnit {
    static constexpr int kWords = BITS == kFp8 ? 4 : 32 % BITS == 0 ? 1 : 3;
    static constexpr int kCodes = 32 * kWords / code_bits(BITS);
};

// Code c of a unit held in w[0 .. kWords): stream bits [b*c, +b).
template <int BITS>
__device__ __forceinline__ uint32_t unit_code(const uint32_t (&w)[GenUnit<BITS>::kWords],
                                              int c) {
    constexpr int B = code_bits(BITS);
    const int pos = B * c, i = pos >> 5, sh = pos & 31;
    const uint32_t v = sh + B <= 32 ? w[i] >> sh : __funnelshift_r(w[i], w[i + 1], sh);
    return v & ((1u << B) - 1u);
}

// Warp reduction of the per-lane sums and the epilogue of one output unit:
// plain, sections with bias, SiLU(gate) * up, or sections with the rotary
// embedding from p.rope_cs; lane m writes token m.
template <int MODE>
__device__ __forceinline__ void gen_finish(const DenseParams &p, int64_t u,
                                           const int64_t (&rows)[2],
                                           float (&acc)[2][kGenTokens], int lane) {
    const int64_t I = p.N / 2;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int m = 0; m < kGenTokens; ++m)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                acc[h][m] += __shfl_xor_sync(0xffffffffu, acc[h][m], o);
    if (lane >= kGenTokens || lane >= p.M) return;
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

template <int BITS, int MODE>
__global__ void __launch_bounds__(kGenThreads)
    qmv_generic_kernel(DenseParams p, int64_t units) {
    constexpr int UW = GenUnit<BITS>::kWords, CU = GenUnit<BITS>::kCodes;
    constexpr bool PAIRS = MODE == 2 || MODE == 3;
    const int lane = threadIdx.x & (kWarp - 1);
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / kWarp;
    const int64_t wpr = (int64_t)p.K * code_bits(BITS) / 32;  // words per row
    const int64_t upr = wpr / UW;                  // code units per row
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
            // a lane takes units ui, ui + 32, ui + 64, ui + 96 per step: four
            // loads (of UW words) in flight, consecutive lanes on consecutive
            // units, and the activations of consecutive lanes contiguous
            // (shorter tails are masked)
            for (int64_t u0 = 0; u0 < upr; u0 += 4 * kWarp) {
                uint32_t words[4][UW];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int64_t ui = u0 + q4 * kWarp + lane;
#pragma unroll
                    for (int j = 0; j < UW; ++j)
                        words[q4][j] = ui < upr ? wrow[ui * UW + j] : 0u;
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int64_t ui = u0 + q4 * kWarp + lane;
                    if (ui >= upr) break;
                    const int64_t k0 = ui * CU;
                    const int g = (int)(k0 >> gshift);  // one group per unit
                    const float s = bf16_bits_to_f32(srow[g]);
                    const float b = bf16_bits_to_f32(brow[g]);
                    float wv[CU];
#pragma unroll
                    for (int c = 0; c < CU; ++c) {
                        // the code's value as a float: an integer as 2^23 + q
                        // minus 2^23 (exact), an fp8 code as its E4M3 number
                        const uint32_t code = unit_code<BITS>(words[q4], c);
                        const float q = BITS == kFp8
                                            ? e4m3_to_f32(code)
                                            : __uint_as_float(0x4b000000u | code) -
                                                  8388608.0f;
                        wv[c] = fmaf(s, q, b);
                    }
#pragma unroll
                    for (int m = 0; m < kGenTokens; ++m) {
                        if (m >= p.M) break;
                        // the unit's CU activations of token m (2 CU bytes)
                        const uint16_t *xm = p.x + (int64_t)m * p.K + k0;
                        if constexpr (CU % 8 == 0) {
#pragma unroll
                            for (int c8 = 0; c8 < CU / 8; ++c8) {
                                const uint4 v = reinterpret_cast<const uint4 *>(xm)[c8];
                                const uint32_t pr[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    acc[h][m] = fmaf(wv[8 * c8 + 2 * e], bf16_lo(pr[e]), acc[h][m]);
                                    acc[h][m] = fmaf(wv[8 * c8 + 2 * e + 1], bf16_hi(pr[e]),
                                                     acc[h][m]);
                                }
                            }
                        } else {
                            const uint32_t *xw = reinterpret_cast<const uint32_t *>(xm);
#pragma unroll
                            for (int c2 = 0; c2 < CU / 2; ++c2) {
                                const uint32_t pr = xw[c2];
                                acc[h][m] = fmaf(wv[2 * c2], bf16_lo(pr), acc[h][m]);
                                acc[h][m] = fmaf(wv[2 * c2 + 1], bf16_hi(pr), acc[h][m]);
                            }
                        }
                    }
                }
            }
        }
        gen_finish<MODE>(p, u, rows, acc, lane);
    }
}

// ------------------------------------------------------------ integer dot
// The same outputs by an exact integer dot, as in the tuned kernels: each
// block first encodes the pass's activations into shared memory as int16
// with a power-of-two scale per weight group (the group's largest magnitude
// maps into [2^14, 2^15)), together with the plain sum of every 32
// activations for the bias term.  A lane takes chunks of 32 codes (a chunk
// never spans two groups: groups are 32, 64 or 128), spreads the chunk's
// codes into eight words of four unsigned bytes and forms sum_k q_k xi_k
// with dp2a (two 16x8-bit products per instruction), so per chunk and token
//   y += (scale * 2^E) * D + bias * sum_k x_k.
// Spreading: widths dividing 8 take byte planes of a word (plane i, the
// word shifted by b*i and masked, holds codes (8/b) j + i in byte j: the
// activations are stored in that order); u3 and u6 spread each run of four
// codes (12 or 24 bits) into the four bytes of a word with shifts and
// masks, keeping the natural order.  Each lane loads 32-64 bytes of codes
// (and the chunks' scales and biases) per step before using any of them.
constexpr int kGdThreads = 512;
constexpr int kGdChunk = 32;  // codes per chunk

template <int BITS>
struct GdFmt {
    static constexpr int CW = kGdChunk * BITS / 32;  // words per chunk
    // chunks per lane and step: 32-64 bytes of codes in flight
    static constexpr int NQ = BITS == 8 || BITS == 6 ? 2 : 4;
};

// Position of code c of a chunk among its activations (dp2a order): within
// each word, byte plane by byte plane for u2 and u4; natural otherwise.
template <int BITS>
__device__ __forceinline__ int gd_pos(int c) {
    if constexpr (BITS == 2 || BITS == 4) {
        constexpr int CPW = 32 / BITS, NP = 8 / BITS;
        const int w = c / CPW, r = c % CPW;
        return w * CPW + 4 * (r % NP) + r / NP;
    } else {
        return c;
    }
}

// A chunk's 32 codes as eight words of four unsigned bytes, in dp2a order.
template <int BITS>
__device__ __forceinline__ void gd_spread(const uint32_t (&w)[GdFmt<BITS>::CW],
                                          uint32_t (&b)[8]) {
    constexpr int CW = GdFmt<BITS>::CW;
    if constexpr (BITS == 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = w[i];
    } else if constexpr (BITS == 4 || BITS == 2) {
        constexpr uint32_t M = BITS == 4 ? 0x0f0f0f0fu : 0x03030303u;
        constexpr int NP = 8 / BITS;
#pragma unroll
        for (int j = 0; j < CW; ++j)
#pragma unroll
            for (int i = 0; i < NP; ++i) b[j * NP + i] = (w[j] >> (BITS * i)) & M;
    } else {
        constexpr int CB = 4 * BITS;  // bits of a run of four codes
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int pos = CB * i, j = pos >> 5, sh = pos & 31;
            const uint32_t v =
                sh + CB <= 32 ? w[j] >> sh
                              : __funnelshift_r(w[j], w[j + 1 < CW ? j + 1 : j], sh);
            if constexpr (BITS == 6)
                b[i] = (v & 0x3fu) | ((v << 2) & 0x3f00u) | ((v << 4) & 0x3f0000u) |
                       ((v << 6) & 0x3f000000u);
            else
                b[i] = (v & 0x7u) | ((v << 5) & 0x700u) | ((v << 10) & 0x70000u) |
                       ((v << 15) & 0x7000000u);
        }
    }
}

// Loads a chunk's CW words (byte offset a multiple of 4 * CW) with the
// widest aligned vectors.
template <int CW>
__device__ __forceinline__ void gd_load(const uint32_t *p, uint32_t (&w)[CW]) {
    if constexpr (CW % 4 == 0) {
#pragma unroll
        for (int i = 0; i < CW / 4; ++i) {
            const uint4 v = reinterpret_cast<const uint4 *>(p)[i];
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    } else if constexpr (CW % 2 == 0) {
#pragma unroll
        for (int i = 0; i < CW / 2; ++i) {
            const uint2 v = reinterpret_cast<const uint2 *>(p)[i];
            w[2 * i] = v.x; w[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < CW; ++i) w[i] = p[i];
    }
}

// Shared bytes of one pass's encoded activations: int16 [M][K], the group
// scales [M][K/group] and the chunk sums [M][K/32].
static size_t gd_smem_bytes(int M, int64_t K, int group) {
    return (size_t)M * (K * 2 + (K / group) * 4 + (K / kGdChunk) * 4);
}

template <int BITS, int MODE>
__global__ void __launch_bounds__(kGdThreads, 2)
    qmv_gdot_kernel(DenseParams p, int64_t units) {
    using F = GdFmt<BITS>;
    constexpr int CW = F::CW, NQ = F::NQ;
    constexpr bool PAIRS = MODE == 2 || MODE == 3;
    constexpr int kWarps = kGdThreads / kWarp;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char gd_smem[];
    const int K = p.K, G = p.G, M = p.M, GS = p.group;
    const int nch = K / kGdChunk;  // chunks per row
    // xe [M][4][nch][8]: the eight activations (dp2a order) of piece s of
    // chunk c at (s * nch + c) * 8, so lanes on consecutive chunks read
    // consecutive 16-byte pieces (no bank conflicts)
    int16_t *xe = reinterpret_cast<int16_t *>(gd_smem);
    float *xf = reinterpret_cast<float *>(gd_smem + (size_t)M * K * 2);  // [M][G]
    float *xu = xf + M * G;                                              // [M][nch]
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x / kWarp;
    const int gshift = __ffs(GS) - 1;  // groups are 32, 64 or 128
    __shared__ int s_mk;  // some group is marked (common.cuh)
    if (threadIdx.x == 0) {
        pdl_launch_dependents();
        s_mk = 0;
    }
    __syncthreads();
    pdl_wait_primary();  // x may be the previous kernel's output

    // encode: one warp per (token, group), four groups' loads in flight; the
    // lane takes inputs lane + 32r of its group, so each r is one chunk
    const int ntask = M * G, rmax = GS / kWarp;
    for (int t0 = warp; t0 < ntask; t0 += 4 * kWarps) {
        float v[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int task = t0 + b * kWarps;
            const int m = task / G, g = task - m * G;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                v[b][r] = task < ntask && r < rmax
                              ? bf16_bits_to_f32(p.x[m * K + g * GS + r * kWarp + lane])
                              : 0.f;
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int task = t0 + b * kWarps;
            if (task >= ntask) break;  // the same for every lane
            const int m = task / G, g = task - m * G;
            int ef = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) ef = max(ef, f32_exp_field(v[b][r]));
            ef = __reduce_max_sync(FULL, ef);
            float f, finv;
            group_scale(ef, f, finv);
            // the group's rounding error and magnitude in units of f; a
            // marked group (common.cuh) keeps raw bf16 in its int16 slots
            float re = 0.f, ab = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                re += i16_resid(v[b][r], finv);
                ab += fabsf(v[b][r]);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                re += __shfl_xor_sync(FULL, re, o);
                ab += __shfl_xor_sync(FULL, ab, o);
            }
            const bool marked = group_marked(re, ab * finv);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r >= rmax) break;
                const int k0 = g * GS + r * kWarp;  // this r's chunk
                const int pos = gd_pos<BITS>(lane);
                xe[m * K + ((pos >> 3) * nch + k0 / kGdChunk) * 8 + (pos & 7)] =
                    marked ? (int16_t)(__float_as_uint(v[b][r]) >> 16)
                           : (int16_t)__float2int_rn(v[b][r] * finv);
                float sum = v[b][r];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
                if (lane == 0) xu[m * nch + k0 / kGdChunk] = sum;
            }
            if (lane == 0) xf[m * G + g] = marked ? -1.f : f;
            if (marked && lane == 0) s_mk = 1;
        }
    }
    __syncthreads();

    const int64_t I = p.N / 2;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    const int64_t nw = (int64_t)gridDim.x * blockDim.x / kWarp;
    const int wpr = K * BITS / 32;  // words per row
    // the unit loop, once with the marked-group path (EX) and once without
    auto unit_loop = [&](auto ex) {
        constexpr bool EX = decltype(ex)::value;
        for (int64_t u = gw; u < units; u += nw) {
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
                const uint16_t *srow = p.sc + rows[h] * G;
                const uint16_t *brow = p.bi + rows[h] * G;
                for (int c0 = 0; c0 < nch; c0 += NQ * kWarp) {
                    // the step's codes, scales and biases (scale | bias << 16),
                    // every load issued before any is used
                    uint32_t words[NQ][CW], sb[NQ];
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const int ci = c0 + q * kWarp + lane;
                        if (ci < nch) {
                            gd_load<CW>(wrow + ci * CW, words[q]);
                            const int g = (ci * kGdChunk) >> gshift;
                            sb[q] = (uint32_t)srow[g] | ((uint32_t)brow[g] << 16);
                        } else {
#pragma unroll
                            for (int j = 0; j < CW; ++j) words[q][j] = 0u;
                            sb[q] = 0u;
                        }
                    }
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const int ci = c0 + q * kWarp + lane;
                        if (ci >= nch) break;
                        const int g = (ci * kGdChunk) >> gshift;
                        const float sc = bf16_lo(sb[q]), bi = bf16_hi(sb[q]);
                        uint32_t bw[8];
                        gd_spread<BITS>(words[q], bw);
#pragma unroll
                        for (int m = 0; m < kGenTokens; ++m) {
                            if (m >= M) break;
                            const uint4 *xp = reinterpret_cast<const uint4 *>(xe + m * K);
                            const float fg = xf[m * G + g];
                            float dq;
                            if (!EX || fg >= 0.f) {
                                int d = 0;
#pragma unroll
                                for (int s4 = 0; s4 < 4; ++s4) {
                                    const uint4 x4 = xp[s4 * nch + ci];
                                    d = dp2a_hi(x4.y, bw[2 * s4], dp2a_lo(x4.x, bw[2 * s4], d));
                                    d = dp2a_hi(x4.w, bw[2 * s4 + 1],
                                                dp2a_lo(x4.z, bw[2 * s4 + 1], d));
                                }
                                dq = fg * (float)d;
                            } else {  // marked group: fp32 dot of the raw activations
                                dq = 0.f;
#pragma unroll
                                for (int s4 = 0; s4 < 4; ++s4) {
                                    const uint4 x4 = xp[s4 * nch + ci];
                                    dq = fdp2a_hi(x4.y, bw[2 * s4], fdp2a_lo(x4.x, bw[2 * s4], dq));
                                    dq = fdp2a_hi(x4.w, bw[2 * s4 + 1],
                                                  fdp2a_lo(x4.z, bw[2 * s4 + 1], dq));
                                }
                            }
                            acc[h][m] = fmaf(sc, dq, fmaf(bi, xu[m * nch + ci], acc[h][m]));
                        }
                    }
                }
            }
            gen_finish<MODE>(p, u, rows, acc, lane);
        }
    };
    if (s_mk)
        unit_loop(std::true_type{});
    else
        unit_loop(std::false_type{});
}

template <int BITS>
static cudaError_t launch_gdot_b(int mode, const DenseParams &p,
                                 cudaStream_t st) {
    const int64_t units = mode == 2 || mode == 3 ? p.N / 2 : p.N;
    if (units <= 0) return cudaSuccess;
    const void *k = mode == 0   ? reinterpret_cast<const void *>(qmv_gdot_kernel<BITS, 0>)
                    : mode == 1 ? reinterpret_cast<const void *>(qmv_gdot_kernel<BITS, 1>)
                    : mode == 2 ? reinterpret_cast<const void *>(qmv_gdot_kernel<BITS, 2>)
                                : reinterpret_cast<const void *>(qmv_gdot_kernel<BITS, 3>);
    const size_t smem = gd_smem_bytes(p.M, p.K, p.group);
    int grid = 0;
    cudaError_t e = occupancy_grid(k, kGdThreads, smem, &grid);
    if (e != cudaSuccess) return e;
    const int64_t need = (units + kGdThreads / kWarp - 1) / (kGdThreads / kWarp);
    if (grid > need) grid = (int)need;
    return launch_pdl(k, (unsigned)grid, (unsigned)kGdThreads, smem, st, p, units);
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
// The integer-dot kernel when the pass's encoded activations fit in shared
// memory (K up to ~16K inputs at four tokens), else the fp32 kernel.
constexpr size_t kGdMaxSmem = 200 * 1024;

template <int BITS>
static cudaError_t launch_generic_w(int mode, const DenseParams &p,
                                    cudaStream_t st) {
    if (gd_smem_bytes(p.M, p.K, p.group) <= kGdMaxSmem)
        return launch_gdot_b<BITS>(mode, p, st);
    return launch_generic_b<BITS>(mode, p, st);
}

cudaError_t launch_generic(int mode, const DenseParams &p, cudaStream_t st) {
    switch (p.bits) {
        case 2: return launch_generic_w<2>(mode, p, st);
        case 3: return launch_generic_w<3>(mode, p, st);
        case 4: return launch_generic_w<4>(mode, p, st);
        case 6: return launch_generic_w<6>(mode, p, st);
        case 8: return launch_generic_w<8>(mode, p, st);
        // fp8 codes: fp32 products (an E4M3 value is no integer)
        case kFp8: return launch_generic_b<kFp8>(mode, p, st);
        default: return cudaErrorInvalidValue;
    }
}

int generic_max_tokens() { return kGenTokens; }

}  // namespace gwa
