/*
 * oracle.c -- plain fp64 CPU reference for MLX-style affine group-quantized
 * projections.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library; both sides see the same seeded inputs and nothing else.
 *
 * What it computes is the plain definition, written out with no blocking,
 * fusion or reordering:
 *
 *   code   q[n,k] = (Wq[n, k/P] >> (b*(k mod P))) & (2^b - 1),  P = 32/b
 *   weight w[n,k] = S[n, k/G] * q[n,k] + B[n, k/G]                (fp64)
 *   output y[m,n] = sum_k x[m,k] * w[n,k]      (fp64, summed in k order)
 *
 * Sources (page title, section):
 *   "Sanctum-MLX", server diagram ("4-bit quantized inference:
 *       QuantizedLinear group_size=64") and the model parameter table
 *       ("Quantization 4-bit, group_size=64").
 *   "The Cathedral Doubled Itself", "The two fusions": the fused QKV weight
 *       is [q_out + 2*kv_out, hidden/8] -- eight 4-bit codes per 32-bit word
 *       along the input axis -- and its one matmul output is split back into
 *       Q, K, V on the last axis; the gate+up fusion applies the same recipe
 *       to gate_proj and up_proj ahead of SiLU and the multiply.
 *   "saragossa", "Quantization formats": MLX affine integer weights
 *       u2/u3/u4/u6/u8 at group size 64 with bf16 scales and biases; u3
 *       ~3.5, u4 ~4.5, u6 ~6.5 and u8 ~8.5 bpw, i.e. two 16-bit parameters
 *       per 64 weights.
 *   "Sanctum-MLX" and "Four Candles For The Cathedral": 3-D switch_mlp expert
 *       grids with per-expert gate_proj / up_proj (MoE routed experts).
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes):
 *   - bit order: a row's words form one little-endian bit stream and code k
 *     sits at its bits [b*k, +b), lowest bits first.  For b dividing 32
 *     (u2, u4, u8) that is field k mod P of word k / P, P = 32/b; a u3 or u6
 *     code may straddle two words (its low bits at the top of one word, the
 *     rest at the bottom of the next);
 *   - codes are unsigned, 0 .. 2^b-1; the affine bias carries any offset;
 *   - the dequantized weight is scale*q + bias;
 *   - gate rows come first, then up rows; SiLU(g) = g / (1 + exp(-g));
 *   - MoE: gate+up mode gives h[t,j,:] = SiLU(Wg[e] x_t) * (Wu[e] x_t) for
 *     e = ids[t,j]; down mode gives y[t,:] = sum_j r[t,j] * (Wd[e] h[t,j,:]),
 *     summed over j in slot order;
 *   - fp8 (e4m3), listed by "saragossa", "Quantization formats" beside the
 *     affine widths with the u8 footprint: 8-bit codes in the same container
 *     (four per word, lowest byte first) whose value is the OCP FP8 E4M3
 *     number of the byte (sign bit 7, exponent bits 6..3 with bias 7,
 *     mantissa bits 2..0; exponent 0: subnormal m/8 * 2^-6; exponent 15 with
 *     mantissa 7: NaN; no infinities), dequantized as scale * value + bias.
 *     Selected by bits = ORC_FP8 (the library's GWA_FP8_E4M3 value, written
 *     out here on its own).
 *
 * bf16 values arrive as their 16-bit patterns; widening bf16 -> fp32 -> fp64
 * is exact.  Compile with -ffp-contract=off so no multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD_ARG (-1)

/* Exact widening of a bf16 bit pattern: the 16 bits are the top half of an
 * IEEE binary32. */
double orc_bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

#define ORC_FP8 0x108

static int bits_ok(int bits) {
    return bits == 2 || bits == 3 || bits == 4 || bits == 6 || bits == 8 ||
           bits == ORC_FP8;
}

/* Bits a code takes in the stream. */
static int code_width(int bits) { return bits == ORC_FP8 ? 8 : bits; }

/* The OCP FP8 E4M3 number of a byte, from its fields. */
double orc_e4m3_value(uint32_t byte) {
    const int sign = (int)((byte >> 7) & 1u);
    const int e = (int)((byte >> 3) & 15u);
    const int m = (int)(byte & 7u);
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The value a code stands for before the affine map: the integer itself,
 * or its E4M3 number. */
static double code_value(uint32_t code, int bits) {
    return bits == ORC_FP8 ? orc_e4m3_value(code) : (double)code;
}

/* The integer code at (row n, input k): bits [b*k, b*k + b) of the row's
 * bit stream, word j holding stream bits [32j, 32j + 32). */
static inline uint32_t code_at(const uint32_t *wq, int64_t words_per_row,
                               int64_t n, int64_t k, int bits) {
    bits = code_width(bits);
    const uint32_t *row = wq + n * words_per_row;
    int64_t pos = (int64_t)bits * k;      /* stream position of the low bit */
    uint32_t shift = (uint32_t)(pos % 32);
    uint32_t code = row[pos / 32] >> shift;
    if (shift + (uint32_t)bits > 32u)     /* the rest in the next word */
        code |= row[pos / 32 + 1] << (32u - shift);
    return code & ((1u << bits) - 1u);
}

/* A row of K codes must fill whole words. */
static int shape_ok(int64_t N, int64_t K, int bits, int group) {
    if (N < 0 || K < 0 || !bits_ok(bits) || group <= 0) return 0;
    if (K % group != 0) return 0;
    if ((K * code_width(bits)) % 32 != 0) return 0;
    return 1;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Step 1 -- unpack: codes[n*K + k] = q[n,k]. */
int orc_unpack(const uint32_t *wq, int64_t N, int64_t K, int bits,
               uint8_t *codes) {
    if (!shape_ok(N, K, bits, 1)) return ORC_BAD_ARG;
    int64_t wpr = K * code_width(bits) / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)code_at(wq, wpr, n, k, bits);
    return ORC_OK;
}

/* Step 2 -- dequantize: w[n*K + k] = S[n,k/G] * q[n,k] + B[n,k/G], fp64. */
int orc_dequant(const uint32_t *wq, const uint16_t *scales,
                const uint16_t *biases, int64_t N, int64_t K, int bits,
                int group, double *w) {
    if (!shape_ok(N, K, bits, group)) return ORC_BAD_ARG;
    int64_t wpr = K * code_width(bits) / 32, gpr = K / group;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            double s = orc_bf16_to_f64(scales[n * gpr + k / group]);
            double b = orc_bf16_to_f64(biases[n * gpr + k / group]);
            double q = code_value(code_at(wq, wpr, n, k, bits), bits);
            w[n * K + k] = s * q + b;
        }
    return ORC_OK;
}

/* One output: sum over k, in k order, of x[k] * (S*q + B). */
static double dot_row(const uint16_t *xrow, const uint32_t *wq,
                      const uint16_t *scales, const uint16_t *biases,
                      int64_t n, int64_t K, int bits, int group) {
    int64_t wpr = K * code_width(bits) / 32, gpr = K / group;
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double s = orc_bf16_to_f64(scales[n * gpr + k / group]);
        double b = orc_bf16_to_f64(biases[n * gpr + k / group]);
        double q = code_value(code_at(wq, wpr, n, k, bits), bits);
        double w = s * q + b;
        acc += orc_bf16_to_f64(xrow[k]) * w;
    }
    return acc;
}

/* Step 3 -- y[m, i] = sum_k x[m,k] * w[rows[i], k] for i < n_rows.
 * rows == NULL means every row 0..N-1 (then n_rows must equal N).
 * x is bf16 [M, K] row-major; y is fp64 [M, n_rows] row-major. */
int orc_qmv(const uint16_t *x, int64_t M, const uint32_t *wq,
            const uint16_t *scales, const uint16_t *biases, int64_t N,
            int64_t K, int bits, int group, const int64_t *rows,
            int64_t n_rows, double *y, int nthreads) {
    if (!shape_ok(N, K, bits, group) || M < 0 || n_rows < 0)
        return ORC_BAD_ARG;
    if (rows == NULL && n_rows != N) return ORC_BAD_ARG;
    for (int64_t i = 0; i < n_rows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= N)) return ORC_BAD_ARG;
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_rows; ++i) {
        int64_t n = rows ? rows[i] : i;
        for (int64_t m = 0; m < M; ++m)
            y[m * n_rows + i] =
                dot_row(x + m * K, wq, scales, biases, n, K, bits, group);
    }
    return ORC_OK;
}

/* SiLU(g) = g / (1 + exp(-g)) in fp64. */
double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* Step 5 -- fused gate+up with the SiLU(gate)*up epilogue.  The weight has
 * 2*I rows: rows [0, I) are gate_proj, rows [I, 2I) are up_proj.
 * h[m, i] = SiLU(g) * u with g = row cols[i] and u = row I + cols[i];
 * cols == NULL means every column 0..I-1. */
int orc_gate_up_silu(const uint16_t *x, int64_t M, const uint32_t *wq,
                     const uint16_t *scales, const uint16_t *biases,
                     int64_t N2, int64_t K, int bits, int group,
                     const int64_t *cols, int64_t n_cols, double *h,
                     int nthreads) {
    if (!shape_ok(N2, K, bits, group) || N2 % 2 != 0 || M < 0)
        return ORC_BAD_ARG;
    int64_t I = N2 / 2;
    if (cols == NULL && n_cols != I) return ORC_BAD_ARG;
    for (int64_t i = 0; i < n_cols; ++i)
        if (cols && (cols[i] < 0 || cols[i] >= I)) return ORC_BAD_ARG;
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n_cols; ++i) {
        int64_t c = cols ? cols[i] : i;
        for (int64_t m = 0; m < M; ++m) {
            double g = dot_row(x + m * K, wq, scales, biases, c, K, bits,
                               group);
            double u = dot_row(x + m * K, wq, scales, biases, I + c, K, bits,
                               group);
            h[m * n_cols + i] = orc_silu(g) * u;
        }
    }
    return ORC_OK;
}

/* Step 6a -- MoE gate+up: stacked expert weights, expert e occupies rows
 * [e*N2, (e+1)*N2) of wq/scales/biases (each expert is a 2*I x K fused
 * gate+up matrix).  h[t, j, i] = SiLU(g) * u for expert ids[t, j];
 * h is fp64 [M, topk, I]. */
int orc_moe_gate_up_silu(const uint16_t *x, int64_t M, int64_t topk,
                         const int32_t *ids, const uint32_t *wq,
                         const uint16_t *scales, const uint16_t *biases,
                         int64_t E, int64_t N2, int64_t K, int bits,
                         int group, double *h, int nthreads) {
    if (!shape_ok(N2, K, bits, group) || N2 % 2 != 0 || M < 0 || topk < 0)
        return ORC_BAD_ARG;
    for (int64_t p = 0; p < M * topk; ++p)
        if (ids[p] < 0 || ids[p] >= E) return ORC_BAD_ARG;
    int64_t I = N2 / 2;
    int64_t wpr = K * code_width(bits) / 32, gpr = K / group;
    set_threads(nthreads);
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t t = 0; t < M; ++t)
        for (int64_t j = 0; j < topk; ++j) {
            int64_t e = ids[t * topk + j];
            const uint32_t *we = wq + e * N2 * wpr;
            const uint16_t *se = scales + e * N2 * gpr;
            const uint16_t *be = biases + e * N2 * gpr;
            for (int64_t i = 0; i < I; ++i) {
                double g = dot_row(x + t * K, we, se, be, i, K, bits, group);
                double u =
                    dot_row(x + t * K, we, se, be, I + i, K, bits, group);
                h[(t * topk + j) * I + i] = orc_silu(g) * u;
            }
        }
    return ORC_OK;
}

/* Step 6b -- MoE down + routed combine.  hin is bf16 [M, topk, K]; expert e
 * occupies rows [e*N, (e+1)*N).  y[t, n] = sum_j r[t,j] * (Wd[e] hin[t,j])[n]
 * with the sum over j in slot order; y is fp64 [M, N]. */
int orc_moe_down_combine(const uint16_t *hin, int64_t M, int64_t topk,
                         const int32_t *ids, const float *route_w,
                         const uint32_t *wq, const uint16_t *scales,
                         const uint16_t *biases, int64_t E, int64_t N,
                         int64_t K, int bits, int group, double *y,
                         int nthreads) {
    if (!shape_ok(N, K, bits, group) || M < 0 || topk < 0) return ORC_BAD_ARG;
    for (int64_t p = 0; p < M * topk; ++p)
        if (ids[p] < 0 || ids[p] >= E) return ORC_BAD_ARG;
    int64_t wpr = K * code_width(bits) / 32, gpr = K / group;
    set_threads(nthreads);
#pragma omp parallel for schedule(static) collapse(2)
    for (int64_t t = 0; t < M; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < topk; ++j) {
                int64_t e = ids[t * topk + j];
                double d = dot_row(hin + (t * topk + j) * K, wq + e * N * wpr,
                                   scales + e * N * gpr, biases + e * N * gpr,
                                   n, K, bits, group);
                acc += (double)route_w[t * topk + j] * d;
            }
            y[t * N + n] = acc;
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Affine quantization, the requantize step of "Sanctum-MLX", "The April 2026
 * cutover" (LoRA merge at load: dequantize, add the delta, requantize at
 * group size 64 and 4 bits; "File map": lora.rs merges quantized and
 * switch_mlp expert weights).  The pages give no rounding rule; the plainest
 * reading, per group of G consecutive inputs of a row:
 *
 *   lo = min w, hi = max w          (the bf16 values, exact in fp32)
 *   s  = bf16_rn((hi - lo) / (2^b - 1))        fp32 subtract, divide (RN)
 *   z  = lo                         (a bf16 value already: stored as is,
 *                                    a zero as +0)
 *   q  = clamp(rint((w - z) / s), 0, 2^b - 1)  fp32, round half to even;
 *        q = 0 for every input when s == 0
 *
 * and the codes are packed lowest bits first, P = 32/b per word.  A code is
 * an integer decided in floating point, so this step runs in the kernel's
 * precision (IEEE fp32, round to nearest even) instead of fp64; both sides
 * then reach the same code.  Inputs must be finite.
 */

/* fp32 -> bf16 bit pattern, round to nearest, ties to even (finite input):
 * add half an ulp of the kept part, plus one when the kept part is odd,
 * then truncate to the top 16 bits. */
static uint16_t f32_to_bf16_rn(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* w: bf16 [N, K]; out wq [N, K*b/32], scales and biases bf16 [N, K/G];
 * widths that divide 32 (u2, u4, u8). */
int orc_quantize_affine(const uint16_t *w, int64_t N, int64_t K, int bits,
                        int group, uint32_t *wq, uint16_t *scales,
                        uint16_t *biases) {
    if (!shape_ok(N, K, bits, group) || 32 % bits != 0) return ORC_BAD_ARG;
    const int64_t gpr = K / group, wpr = K * bits / 32;
    const int per_word = 32 / bits;
    const uint32_t qmax = (1u << bits) - 1u;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t w0 = 0; w0 < wpr; ++w0) wq[n * wpr + w0] = 0u;
        for (int64_t g = 0; g < gpr; ++g) {
            const uint16_t *src = w + n * K + g * group;
            float lo = bf16_to_f32(src[0]), hi = lo;
            for (int i = 1; i < group; ++i) {
                const float v = bf16_to_f32(src[i]);
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            /* a minimum of zero is stored as +0 whichever zeros occur
             * (-0 + +0 = +0 in round to nearest) */
            lo = lo + 0.0f;
            const float range = hi - lo;
            const uint16_t sbits = f32_to_bf16_rn(range / (float)qmax);
            const float s = bf16_to_f32(sbits);
            uint16_t zbits;
            {
                uint32_t u;
                memcpy(&u, &lo, sizeof u);
                zbits = (uint16_t)(u >> 16);
            }
            scales[n * gpr + g] = sbits;
            biases[n * gpr + g] = zbits;
            for (int i = 0; i < group; ++i) {
                uint32_t q = 0u;
                if (s != 0.0f) {
                    const float t = rintf((bf16_to_f32(src[i]) - lo) / s);
                    q = t <= 0.0f ? 0u : t >= (float)qmax ? qmax : (uint32_t)t;
                }
                const int64_t k = g * group + i;
                wq[n * wpr + k / per_word] |=
                    q << (uint32_t)(bits * (k % per_word));
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Rotary position embedding of the fused QKV output ("The Cathedral Doubled
 * Itself", "The kernel that worked and the kernel that won't": the next step
 * after the fused projection is a kernel that also applies RoPE to the
 * materialized Q and K, which the pages designed but did not ship; "The trap
 * that ate three hours": RoPE consumes Q and K per head at the cache offset).
 * The pages give no formula; the textbook form with the rotate-half pairing
 * (element i of a head with element i + d/2):
 *
 *   theta_i = pos * base^(-2i/d),  i = 0 .. d/2 - 1
 *   y'[i]       = y[i] cos theta_i - y[i + d/2] sin theta_i
 *   y'[i + d/2] = y[i + d/2] cos theta_i + y[i] sin theta_i
 *
 * for every head of Q and of K (d = head_dim), in place on fp64 rows;
 * pos = positions[m] for token m.  V is not rotated.
 */
int orc_rope(double *y, int64_t M, int64_t width, int64_t head_dim,
             double base, const int32_t *positions) {
    if (M < 0 || width < 0 || head_dim <= 0 || head_dim % 2 != 0 ||
        width % head_dim != 0 || !(base > 0.0))
        return ORC_BAD_ARG;
    const int64_t half = head_dim / 2;
    for (int64_t m = 0; m < M; ++m) {
        const double pos = (double)positions[m];
        for (int64_t h = 0; h < width / head_dim; ++h) {
            double *row = y + m * width + h * head_dim;
            for (int64_t i = 0; i < half; ++i) {
                const double theta =
                    pos * pow(base, -2.0 * (double)i / (double)head_dim);
                const double c = cos(theta), sn = sin(theta);
                const double a = row[i], b = row[i + half];
                row[i] = a * c - b * sn;
                row[i + half] = b * c + a * sn;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Attention with a 4-bit value cache ("Sanctum-MLX", the six-changes table,
 * row 5 "Fused attention with inline V dequant (sdpa_dequant_v)", and the
 * paragraph after it: Q, a materialized bf16 K and the compressed V state
 * (indices, scales, zeros) in; SDPA with V dequantized inline, causal mask,
 * GQA without copies; "File map": turboquant/ holds the 4-bit value cache).
 * The pages do not print the value format; the reading here is this
 * library's affine format along the head dimension: codes of `bits` bits
 * packed 32/bits per word, one bf16 scale and bias ("zero") per `group`
 * values, v = scale * q + bias.  Plain softmax attention in fp64:
 *
 *   score[t] = scale * sum_d q[d] k[t][d]
 *   p[t]     = exp(score[t] - max) / sum_t' exp(score[t'] - max)
 *   out[d]   = sum_t p[t] v[t][d]
 *
 * over the keys a query may see: all T, or with the causal mask t <= T - Lq
 * + l for query l of Lq (the queries are the last Lq positions).  Layouts:
 * q [B, Hq, Lq, D], k [B, Hkv, T, D] (bf16), v codes [B, Hkv, T, D*bits/32],
 * v scales / biases [B, Hkv, T, D/group], out [B, Hq, Lq, D] (fp64); query
 * head h reads KV head h / (Hq / Hkv).
 */
int orc_sdpa_dequant_v(const uint16_t *q, int64_t B, int64_t Hq, int64_t Lq,
                       int64_t D, const uint16_t *k, int64_t Hkv, int64_t T,
                       const uint32_t *vq, const uint16_t *vs,
                       const uint16_t *vb, int bits, int group, double scale,
                       int causal, double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Lq < 0 || D <= 0 ||
        T < 0 || !bits_ok(bits) || bits == ORC_FP8 || group <= 0 ||
        D % group != 0 || D % (32 / bits) != 0 || (causal && Lq > T))
        return ORC_BAD_ARG;
    const int64_t rep = Hq / Hkv, wpr = D * bits / 32, gpr = D / group;
    double *p = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    if (!p) return ORC_BAD_ARG;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < Hq; ++h) {
            const int64_t hk = h / rep;
            const int64_t kv = (b * Hkv + hk) * T;  /* first key row */
            for (int64_t l = 0; l < Lq; ++l) {
                const uint16_t *qv = q + ((b * Hq + h) * Lq + l) * D;
                double *o = out + ((b * Hq + h) * Lq + l) * D;
                const int64_t tn = causal ? T - Lq + l + 1 : T;
                double mx = -INFINITY;
                for (int64_t t = 0; t < tn; ++t) {
                    double sdot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        sdot += orc_bf16_to_f64(qv[d]) *
                                orc_bf16_to_f64(k[(kv + t) * D + d]);
                    p[t] = scale * sdot;
                    if (p[t] > mx) mx = p[t];
                }
                double sum = 0.0;
                for (int64_t t = 0; t < tn; ++t) {
                    p[t] = exp(p[t] - mx);
                    sum += p[t];
                }
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t t = 0; t < tn; ++t) {
                    const int64_t row = kv + t;
                    for (int64_t d = 0; d < D; ++d) {
                        const double sv = orc_bf16_to_f64(vs[row * gpr + d / group]);
                        const double bv = orc_bf16_to_f64(vb[row * gpr + d / group]);
                        const double c = (double)code_at(vq, wpr, row, d, bits);
                        o[d] += p[t] / sum * (sv * c + bv);
                    }
                }
            }
        }
    free(p);
    return ORC_OK;
}

