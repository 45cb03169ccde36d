// Streaming decode kernels (M <= 4): the weight rows a CTA owns are copied
// into a shared-memory ring by the bulk-copy engine while the consumer
// threads compute, so HBM sees a deep queue of large contiguous reads and the
// consumers never wait on a per-thread load.
//
// Layout of the work:
//  * Units (rows, or gate/up row pairs) are split evenly over the CTAs: CTA i
//    owns units [U*i/grid, U*(i+1)/grid).  Every SM gets the same number of
//    bytes to stream whatever N is.
//  * One producer thread issues, per stage, contiguous bulk copies of the
//    stage's packed rows and their scales and biases (a row's bytes are
//    contiguous in the packed format, and so are consecutive rows).
//  * Consumer thread t owns 16-byte chunk t of every row.  It keeps the
//    activations of that chunk (int16-encoded per group, see common.cuh)
//    in registers for the whole kernel, so shared memory only carries the
//    weights.  Per stage it forms the exact integer dot of its chunk for
//    each row and scales it, reduces the rows across the warp with one
//    transpose reduction, and stores the warp totals in per-warp slots that
//    the epilogue adds in a fixed order.
//  * After the last stage the CTA writes its rows: plain output, section
//    buffers, or SiLU(gate)*up.
// Formulas and sources as in qmv.cu ("Sanctum-MLX"; "The Cathedral Doubled
// Itself", "The two fusions"; "saragossa", "Quantization formats").
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gwa {

// fp8 (e4m3) codes: bytes, like u8.
template <>
struct Fmt<kFp8> {
    static constexpr int kCodesPerWord = 4;
    static constexpr int kChunkCodes = 16;
};

static __device__ unsigned int g_stream_timeouts;

// Modes as the host passes them (a plain projection runs as one section).
// kSRope: QKV sections with the rotary embedding, pairs of rows
// (i, i + d/2) of a head (rope_pair_row) laid out like gate/up pairs, in
// stages of whole pairs within one head; the epilogue rotates with the
// (cos, sin) table p.rope_cs.
enum StreamMode { kSPlain = 0, kSSections = 1, kSGateUp = 2, kSRope = 3 };

// A thread's activations for its chunk, encoded for the integer dot (see
// common.cuh): int16 pairs in dp2a order, the group scale 2^E and the plain
// fp32 sum of the chunk's activations.  The chunk's int8 residual planes
// (two-plane path) stay in shared memory, read only by a warp that needs
// them, so that the one-plane loop keeps its registers.
template <int BITS, int MT>
struct XRegs {
    static constexpr int CODES = Fmt<BITS>::kChunkCodes;
    uint32_t pr[MT][CODES / 2];
    float f[MT];
    float xs[MT];
    bool mk[MT];                 // marked group (common.cuh, "marked groups")
};

// Residual plane words of a thread per token and code word: two for u4
// (the entries of the word's low nibbles' inputs, then of its high ones'),
// one for u8, none for fp8 (no integer encoding).  Layout in shared memory:
// [token][code word][thread], so the threads of a warp read consecutive
// words.
template <int BITS>
constexpr int kPlaneWords = BITS == 4 ? 2 : BITS == 8 ? 1 : 0;
template <int BITS>
__device__ __forceinline__ uint2 plane_load(const uint32_t *plane, int pstride,
                                            int m, int wd, int t) {
    const int i = (m * 4 + wd) * pstride + t;
    if constexpr (BITS == 4)
        return reinterpret_cast<const uint2 *>(plane)[i];
    else
        return make_uint2(plane[i], 0u);
}

// Loads and encodes chunk c of each token, and writes the chunk's residual
// planes for thread t (zero unless marked) to `plane`.  Every lane of the
// warp must call this (the lanes of one group agree on its scale and mark
// through shuffles); inactive lanes encode zeros.
template <int BITS, int MT>
__device__ __forceinline__ void load_x_regs(const uint16_t *__restrict__ x,
                                            int M, int K, int c, bool active,
                                            XRegs<BITS, MT> &xr,
                                            uint32_t *plane, int pstride,
                                            int t) {
    constexpr int CODES = Fmt<BITS>::kChunkCodes;
    constexpr int CPG = kGroup / CODES;  // lanes sharing a group
    if constexpr (BITS == kFp8) {
        // fp8: the raw bf16 pairs (fp32 products, no encoding) and the sum
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            uint4 u[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            if (active && m < M) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    x + (int64_t)m * K + (int64_t)c * CODES);
                u[0] = src[0];
                u[1] = src[1];
            }
            const uint32_t w8[8] = {u[0].x, u[0].y, u[0].z, u[0].w,
                                    u[1].x, u[1].y, u[1].z, u[1].w};
            float xs = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                xr.pr[m][i] = w8[i];
                xs += bf16_lo(w8[i]) + bf16_hi(w8[i]);
            }
            xr.f[m] = 1.f;
            xr.mk[m] = false;
            xr.xs[m] = xs;
        }
        return;
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float v[CODES];
        if (active && m < M) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                x + (int64_t)m * K + (int64_t)c * CODES);
#pragma unroll
            for (int i = 0; i < CODES / 8; ++i) {
                const uint4 u = src[i];
                v[8 * i + 0] = bf16_lo(u.x);
                v[8 * i + 1] = bf16_hi(u.x);
                v[8 * i + 2] = bf16_lo(u.y);
                v[8 * i + 3] = bf16_hi(u.y);
                v[8 * i + 4] = bf16_lo(u.z);
                v[8 * i + 5] = bf16_hi(u.z);
                v[8 * i + 6] = bf16_lo(u.w);
                v[8 * i + 7] = bf16_hi(u.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < CODES; ++i) v[i] = 0.f;
        }
        int ef = 0;
#pragma unroll
        for (int i = 0; i < CODES; ++i) ef = max(ef, f32_exp_field(v[i]));
#pragma unroll
        for (int o = 1; o < CPG; o <<= 1)
            ef = max(ef, __shfl_xor_sync(0xffffffffu, ef, o));
        float f, finv;
        group_scale(ef, f, finv);
        float xs = 0.f;
#pragma unroll
        for (int i = 0; i < CODES; ++i) xs += v[i];
        // the group's rounding error and magnitude in units of f
        float re = 0.f, ab = 0.f;
#pragma unroll
        for (int i = 0; i < CODES; ++i) {
            re += i16_resid(v[i], finv);
            ab += fabsf(v[i]);
        }
#pragma unroll
        for (int o = 1; o < CPG; o <<= 1) {
            re += __shfl_xor_sync(0xffffffffu, re, o);
            ab += __shfl_xor_sync(0xffffffffu, ab, o);
        }
        const bool marked = group_marked(re, ab * finv);
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            if constexpr (BITS == 4) {
                uint32_t t[4];
                u4_pairs(v + 8 * wd, finv, t);
#pragma unroll
                for (int i = 0; i < 4; ++i) xr.pr[m][4 * wd + i] = t[i];
            } else {
                uint32_t t[2];
                u8_pairs(v + 4 * wd, finv, t);
                xr.pr[m][2 * wd] = t[0];
                xr.pr[m][2 * wd + 1] = t[1];
            }
        }
        xr.f[m] = f;
        xr.mk[m] = marked;
        xr.xs[m] = xs;
    }
    // The residual planes (zero unless marked), in a second pass that
    // reloads a marked chunk, so that no token's activations stay live
    // beside another's pairs: per u4 word the entries of its low nibbles'
    // inputs (x0 x2 x4 x6), then of its high ones'; per u8 word x0..x3.
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        uint32_t q[CODES / 4];
#pragma unroll
        for (int i = 0; i < CODES / 4; ++i) q[i] = 0u;
        if (xr.mk[m]) {  // marked implies active and m < M
            const float finv = 1.0f / xr.f[m];  // a power of two: exact
            const uint4 *src = reinterpret_cast<const uint4 *>(
                x + (int64_t)m * K + (int64_t)c * CODES);
#pragma unroll
            for (int j = 0; j < CODES / 8; ++j) {
                const uint4 u = src[j];
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
                uint32_t e[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    e[2 * k] = i8_resid(bf16_lo(wv[k]), finv);
                    e[2 * k + 1] = i8_resid(bf16_hi(wv[k]), finv);
                }
                // inputs 8j .. 8j + 7: u4 word j (two plane words), u8
                // words 2j, 2j + 1
                if constexpr (BITS == 4) {
                    q[2 * j] = e[0] | (e[2] << 8) | (e[4] << 16) | (e[6] << 24);
                    q[2 * j + 1] = e[1] | (e[3] << 8) | (e[5] << 16) | (e[7] << 24);
                } else {
                    q[2 * j] = e[0] | (e[1] << 8) | (e[2] << 16) | (e[3] << 24);
                    q[2 * j + 1] = e[4] | (e[5] << 8) | (e[6] << 16) | (e[7] << 24);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < CODES / 4; ++i) {
            // word i: code word i / 2, half i % 2 (u4); code word i (u8)
            const int wd = BITS == 4 ? i >> 1 : i;
            plane[((m * 4 + wd) * pstride + t) * kPlaneWords<BITS> +
                  (BITS == 4 ? (i & 1) : 0)] = q[i];
        }
    }
}

// Chunk dots of R rows against MT tokens: exact integer sums per chunk,
// then (s * 2^E) * D + b * sum(x) in fp32.  The word loop is outside the row
// loop so the rows' dp2a chains interleave; a word's code bytes are split
// once and reused for every token.
template <int BITS, int MT, int R>
__device__ __forceinline__ void batch_dot(const uint4 (&w)[R],
                                          const float (&s)[R],
                                          const float (&b)[R],
                                          const XRegs<BITS, MT> &xr,
                                          float (&out)[R][MT]) {
    if constexpr (BITS == kFp8) {
        // each code's E4M3 value (hardware e4m3 -> fp16 pairs) times the raw
        // bf16 activations, in fp32 (every product exact)
        float2 a[R][MT];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) a[r][m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t word = wd == 0   ? w[r].x
                                      : wd == 1 ? w[r].y
                                      : wd == 2 ? w[r].z
                                                : w[r].w;
                const __half2 h01 = __half2(__nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>(word & 0xffffu), __NV_E4M3));
                const __half2 h23 = __half2(__nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>(word >> 16), __NV_E4M3));
                const float2 q01 = __half22float2(h01), q23 = __half22float2(h23);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t x01 = xr.pr[m][2 * wd], x23 = xr.pr[m][2 * wd + 1];
                    a[r][m] = __ffma2_rn(q01, make_float2(bf16_lo(x01), bf16_hi(x01)),
                                         a[r][m]);
                    a[r][m] = __ffma2_rn(q23, make_float2(bf16_lo(x23), bf16_hi(x23)),
                                         a[r][m]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                out[r][m] = fmaf(s[r], a[r][m].x + a[r][m].y, b[r] * xr.xs[m]);
        return;
    }
    int d[R][MT][2];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) d[r][m][0] = d[r][m][1] = 0;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t word = wd == 0   ? w[r].x
                                  : wd == 1 ? w[r].y
                                  : wd == 2 ? w[r].z
                                            : w[r].w;
            if constexpr (BITS == 4) {
                // high nibbles stay in place (16 * q) and are summed apart
                const uint32_t lo = word & 0x0f0f0f0fu;
                const uint32_t hi = word & 0xf0f0f0f0u;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = xr.pr[m] + 4 * wd;
                    d[r][m][0] = dp2a_hi(pr[1], lo, dp2a_lo(pr[0], lo, d[r][m][0]));
                    d[r][m][1] = dp2a_hi(pr[3], hi, dp2a_lo(pr[2], hi, d[r][m][1]));
                }
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = xr.pr[m] + 2 * wd;
                    int a = d[r][m][wd & 1];
                    a = dp2a_lo(pr[0], word, a);
                    d[r][m][wd & 1] = dp2a_hi(pr[1], word, a);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            // u4: the high-nibble sum is 16x the true sum, exactly
            const int dsum = BITS == 4 ? d[r][m][0] + (d[r][m][1] >> 4)
                                       : d[r][m][0] + d[r][m][1];
            out[r][m] = fmaf(s[r] * xr.f[m], (float)dsum, b[r] * xr.xs[m]);
        }
}

// The residual planes' share of the same chunk dots (two-plane path,
// common.cuh "marked groups"; zero for unmarked groups), 2^-7 of the
// scale, added to out.  A pass of its own, taken only by a warp with a
// marked group, after batch_dot so that the two sets of accumulators are
// never live together; the code words are read again from the stage (the
// slot is still held) and the plane words from shared memory.  Rows go in
// blocks of RB, so that two tokens' u4 accumulators and plane words fit
// beside their pairs.
template <int BITS, int MT, int R>
__device__ __forceinline__ void batch_res(const float (&s)[R],
                                       const XRegs<BITS, MT> &xr,
                                       const unsigned char *base,
                                       const uint32_t (&offw)[R],
                                       const uint32_t *plane, int pstride,
                                       int t, float (&out)[R][MT]) {
    if constexpr (BITS == kFp8) return;  // never marked
    constexpr int RB = (BITS == 4 && MT == 2) ? 1 : R;
#pragma unroll
    for (int r0 = 0; r0 < R; r0 += RB) {
        int e[RB][MT];
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) e[r][m] = 0;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint2 lo = plane_load<BITS>(plane, pstride, m, wd, t);
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const uint32_t word = reinterpret_cast<const uint32_t *>(
                        base + offw[r0 + r])[wd];
                    if constexpr (BITS == 4) {
                        // the high nibbles' products in place (16x), then
                        // the low ones' scaled to match
                        const int h = dp4a_us(word & 0xf0f0f0f0u, lo.y, 0);
                        e[r][m] = dp4a_us(word & 0x0f0f0f0fu, lo.x,
                                          e[r][m] + (h >> 4));
                    } else {
                        e[r][m] = dp4a_us(word, lo.x, e[r][m]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
                out[r0 + r][m] = fmaf(s[r0 + r] * xr.f[m] * 0.0078125f,
                                      (float)e[r][m], out[r0 + r][m]);
    }
}

// Sum of the per-warp slots of one output, in a fixed order.
__device__ __forceinline__ float red_total(const float *red, int idx, int nwh) {
    float t = 0.f;
    for (int w = 0; w < nwh; ++w) t += red[idx * nwh + w];
    return t;
}

// A stage holds UPS = RS * UPT units (rows, or gate/up row pairs); the
// consumer threads form RS row groups, each owning UPT units of the stage
// (RPH = 4 weight rows), and within a group thread c owns chunk c.  Grid:
// one CTA per SM with a ~96 KB ring, so that the next kernel's CTA fits
// beside it and prefetches its first stages while this one drains (2 CTAs
// per SM, 2 or 8 rows per thread and up to 20 consumer warps were measured
// and were slower on the 48-layer stack).
constexpr int kRowsPerThread = 4;

// Registers: up to two tokens, 80 per thread, so that two CTAs of 352 threads
// (rows of 5120 inputs: this kernel and the next one in the stream) share an
// SM (each scheduler's quarter of the register file holds 6 warps of 80);
// four tokens need more and run one CTA per SM.
template <int BITS, int MT, int MODE, int RPH>
__global__ void __maxnreg__(MT == 4 ? 128 : 80)
    qmv_stream_kernel(DenseParams p, int stages, int64_t units, int rs,
                      uint32_t plane_off) {
    constexpr int HALVES = (MODE == kSGateUp || MODE == kSRope) ? 2 : 1;
    constexpr int UPT = RPH / HALVES;     // units per thread per stage
    constexpr int V = RPH * MT;           // values reduced per warp per stage
    constexpr int CODES = Fmt<BITS>::kChunkCodes;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int ncons = blockDim.x - kWarp;
    const int ncpad = ncons / rs;          // threads per row group
    const int nwh = ncpad / kWarp;         // warps per row group
    const int lane = tid & (kWarp - 1);
    const int ups = rs * UPT;              // units per stage
    const uint32_t rowbytes = (uint32_t)p.K * code_bits(BITS) / 8;
    const uint32_t sbrow = (uint32_t)p.G * 2;
    const uint32_t rows_stage = (uint32_t)(HALVES * ups);
    const uint32_t stage_bytes = rows_stage * (rowbytes + 2 * sbrow);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    uint64_t *empty = full + stages;
    float *red = reinterpret_cast<float *>(empty + stages);
    __shared__ int s_issued, s_consumed;

    // rope: whole stages per CTA (ups divides d/2), so no stage crosses a head
    const int64_t ualign = MODE == kSRope ? ups : 1;
    const int64_t u0 = units / ualign * blockIdx.x / gridDim.x * ualign;
    const int64_t u1 = units / ualign * (blockIdx.x + 1) / gridDim.x * ualign;
    const int nu = (int)(u1 - u0);
    const int nst = (nu + ups - 1) / ups;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], ncons / kWarp);
        }
        fence_mbar_init();
        s_issued = 0;
        s_consumed = nst;
        // let the next kernel in the stream start its own weight prefetch
        pdl_launch_dependents();
    }
    __syncthreads();

    if (tid >= ncons) {
        // ------------------------------------------------ producer
        if (tid == ncons) {
            const unsigned char *wq =
                reinterpret_cast<const unsigned char *>(p.wq);
            const unsigned char *sc =
                reinterpret_cast<const unsigned char *>(p.sc);
            const unsigned char *bi =
                reinterpret_cast<const unsigned char *>(p.bi);
            for (int st = 0; st < nst; ++st) {
                const int s = st % stages;
                // Weights are never written by this library's kernels, and a
                // kernel of any other kind completes before one of ours starts
                // (it never triggers an early launch), so the first `stages`
                // stages can be fetched before the previous grid finishes.
                if (st == stages) pdl_wait_primary();
                if (st >= stages &&
                    !mbar_wait(&empty[s], ((st / stages) & 1) ^ 1)) {
                    atomicAdd(&g_stream_timeouts, 1u);
                    break;
                }
                const int64_t ua = u0 + (int64_t)st * ups;
                const int n = (int)min((int64_t)ups, u1 - ua);
                unsigned char *base = smem + (size_t)s * stage_bytes;
                unsigned char *dsc = base + rows_stage * rowbytes;
                unsigned char *dbi = dsc + rows_stage * sbrow;
                mbar_expect_tx(&full[s], (uint32_t)(HALVES * n) *
                                             (rowbytes + 2 * sbrow));
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    const int64_t r = MODE == kSRope
                                          ? rope_pair_row(ua, h, p.rope_hd)
                                          : ua + (h ? p.I : 0);
                    bulk_g2s(base + h * ups * rowbytes, wq + r * rowbytes,
                             n * rowbytes, &full[s]);
                    bulk_g2s(dsc + h * ups * sbrow, sc + r * sbrow, n * sbrow,
                             &full[s]);
                    bulk_g2s(dbi + h * ups * sbrow, bi + r * sbrow, n * sbrow,
                             &full[s]);
                }
                s_issued = st + 1;
            }
        }
    } else {
        // ------------------------------------------------ consumers
        const int hg = tid / ncpad;          // row group
        const int c = tid - hg * ncpad;      // chunk
        const int wh = c / kWarp;            // warp within the row group
        const bool active = c < p.nch;
        // lanes past the row end use chunk 0 (and its group) with zero
        // activations, so every value they read is a finite weight
        const int cc = active ? c : 0;
        const int g = (cc * CODES) / kGroup;
        XRegs<BITS, MT> xr;
        uint32_t *plane = reinterpret_cast<uint32_t *>(smem + plane_off);
        pdl_wait_primary();  // x may be the previous kernel's output
        load_x_regs<BITS, MT>(p.x, p.M, p.K, c, active, xr, plane, ncons, tid);
        // This thread's rows are unit hg*UPT + u of each half of a stage;
        // their shared-memory offsets are the same in every stage.  Row
        // slots past the stage end hold stale data; their totals are
        // dropped below.
        uint32_t offw[RPH], offs[RPH];
        const uint32_t sb_delta = rows_stage * (uint32_t)p.G * 2u;
#pragma unroll
        for (int j = 0; j < RPH; ++j) {
            const uint32_t srow =
                (uint32_t)((j / UPT) * ups + hg * UPT + (j % UPT));
            offw[j] = srow * rowbytes + (uint32_t)cc * 16u;
            offs[j] = rows_stage * rowbytes + (srow * (uint32_t)p.G + g) * 2u;
        }
        // A warp none of whose lanes holds a marked group runs the one-plane
        // copy of the stage loop.
        bool anymk = false;
#pragma unroll
        for (int m = 0; m < MT; ++m) anymk |= xr.mk[m];
        // The stage loop, once with the residual-plane pass (EX) and once
        // without it, so that each copy gets its own register allocation.
        auto stage_loop = [&](auto ex) {
            constexpr bool EX = decltype(ex)::value;
            for (int st = 0; st < nst; ++st) {
                const int s = st % stages;
                if (!mbar_wait(&full[s], (st / stages) & 1)) {
                    atomicAdd(&g_stream_timeouts, 1u);
                    atomicMin(&s_consumed, st);
                    break;
                }
                const int64_t ua = u0 + (int64_t)st * ups;
                const int n = (int)min((int64_t)ups, u1 - ua);
                const unsigned char *base = smem + (uint32_t)s * stage_bytes;
                uint4 w[RPH];
                float sv[RPH], bv[RPH];
#pragma unroll
                for (int j = 0; j < RPH; ++j) {
                    w[j] = *reinterpret_cast<const uint4 *>(base + offw[j]);
                    sv[j] = bf16_bits_to_f32(
                        *reinterpret_cast<const uint16_t *>(base + offs[j]));
                    bv[j] = bf16_bits_to_f32(*reinterpret_cast<const uint16_t *>(
                        base + offs[j] + sb_delta));
                }
                float o[RPH][MT];
                batch_dot<BITS, MT, RPH>(w, sv, bv, xr, o);
                if constexpr (EX)
                    batch_res<BITS, MT, RPH>(sv, xr, base, offw, plane, ncons,
                                             tid, o);
                float v[V];
#pragma unroll
                for (int j = 0; j < RPH; ++j)
#pragma unroll
                    for (int m = 0; m < MT; ++m) v[j * MT + m] = o[j][m];
                // every lane's reads of this stage are done: release the slot
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                const float tot = transpose_reduce<V>(v, lane);
                constexpr int SPREAD = kWarp / V;
                if ((lane & (SPREAD - 1)) == 0) {
                    const int idx = lane / SPREAD;  // j * MT + m
                    const int j = idx / MT, m = idx % MT;
                    const int u = hg * UPT + (j % UPT), h = j / UPT;
                    // per-warp slot: the epilogue adds the warps in a fixed order
                    if (u < n)
                        red[((((st * ups + u) * HALVES + h) * MT + m) * nwh) + wh] =
                            tot;
                }
            }
        };
        if (__any_sync(0xffffffffu, anymk))
            stage_loop(std::true_type{});
        else
            stage_loop(std::false_type{});
    }
    __syncthreads();
    pdl_wait_primary();  // outputs may alias the previous kernel's inputs
    // A timed-out pipeline must not leave bulk copies landing in shared
    // memory after the CTA exits: wait (again bounded) for every stage that
    // was issued but not consumed.
    if (tid == ncons && s_consumed < s_issued) {
        for (int st = s_consumed; st < s_issued; ++st)
            if (!mbar_wait(&full[st % stages], (st / stages) & 1)) break;
    }
    __syncthreads();

    // ---------------------------------------------------- epilogue
    for (int i = tid; i < nu * MT; i += blockDim.x) {
        const int lu = i / MT, m = i % MT;
        if (m >= p.M) continue;
        const int64_t n = u0 + lu;
        if constexpr (MODE == kSGateUp) {
            const float gv = red_total(red, (lu * 2 + 0) * MT + m, nwh);
            const float uv = red_total(red, (lu * 2 + 1) * MT + m, nwh);
            p.y[(int64_t)m * p.I + n] = f32_to_bf16_bits(
                gv / (1.0f + __expf(-gv)) * uv);
        } else if constexpr (MODE == kSRope) {
            const int half = p.rope_hd / 2;
            float a = red_total(red, (lu * 2 + 0) * MT + m, nwh);
            float b = red_total(red, (lu * 2 + 1) * MT + m, nwh);
            const int64_t r0 = rope_pair_row(n, 0, p.rope_hd);
            int s = 0;
            while (s + 1 < p.nsec && r0 >= p.sec_start[s + 1]) ++s;
            const int64_t j = r0 - p.sec_start[s];
            const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
            if (p.sec_bias[s]) {
                a += bf16_bits_to_f32(p.sec_bias[s][j]);
                b += bf16_bits_to_f32(p.sec_bias[s][j + half]);
            }
            if (r0 < p.rope_end) {
                const float2 t = p.rope_cs[(int64_t)m * half + (int)(n % half)];
                const float a2 = a * t.x - b * t.y;
                b = b * t.x + a * t.y;
                a = a2;
            }
            uint16_t *o = p.sec_out[s] + (int64_t)m * size + j;
            o[0] = f32_to_bf16_bits(a);
            o[half] = f32_to_bf16_bits(b);
        } else {
            int s = 0;
            while (s + 1 < p.nsec && n >= p.sec_start[s + 1]) ++s;
            const int64_t j = n - p.sec_start[s];
            const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
            float val = red_total(red, lu * MT + m, nwh);
            if (p.sec_bias[s]) val += bf16_bits_to_f32(p.sec_bias[s][j]);
            p.sec_out[s][(int64_t)m * size + j] = f32_to_bf16_bits(val);
        }
    }
}

// ------------------------------------------------------------ host side
template <int BITS, int MT, int MODE, int RPH>
static cudaError_t launch_stream_r(const DenseParams &p, cudaStream_t st,
                                   bool *used) {
    constexpr int HALVES = (MODE == kSGateUp || MODE == kSRope) ? 2 : 1;
    constexpr int UPT = RPH / HALVES;
    const int64_t units =
        MODE == kSGateUp ? p.I : MODE == kSRope ? p.N / 2 : p.N;
    const size_t rowbytes = (size_t)p.K * code_bits(BITS) / 8;
    const size_t sbrow = (size_t)p.G * 2;
    const int nwh = (p.nch + kWarp - 1) / kWarp;
    // row groups: aim for about ten consumer warps per CTA
    int rs = 1;
    while (rs < 4 && nwh * rs * 2 <= 12) rs *= 2;
    const int threads = nwh * kWarp * rs + kWarp;
    if (threads > kStreamMaxThreads) return cudaSuccess;  // not used
    if (MODE == kSRope && ((p.rope_hd / 2) % (rs * UPT)) != 0)
        return cudaSuccess;  // not used: stages would cross heads
    const size_t stage_bytes = (size_t)HALVES * rs * UPT * (rowbytes + 2 * sbrow);
    int stages = (int)(kStreamRingTarget / stage_bytes);
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    // one CTA per SM, so the next kernel's CTA fits beside it and can
    // prefetch while this one drains
    int grid = num_sms();
    if ((int64_t)grid > units) grid = (int)units;
    // units per CTA, at most (rope: plus one stage for the alignment)
    const int64_t umax =
        (units + grid - 1) / grid + (MODE == kSRope ? rs * UPT : 0);
    const size_t red_bytes = (size_t)umax * HALVES * MT * 4 * nwh;
    // residual planes: per consumer thread and token, 8 (u4) or 4 (u8) words
    const size_t ncons = (size_t)threads - kWarp;
    const size_t plane_off =
        (stages * stage_bytes + 16 * stages + red_bytes + 15) / 16 * 16;
    const size_t smem = plane_off + ncons * MT * 4 * kPlaneWords<BITS> * 4;
    if (smem > kMaxDynSmem) return cudaSuccess;
    auto kern = qmv_stream_kernel<BITS, MT, MODE, RPH>;
    int dummy = 0;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   threads, smem, &dummy);
    if (e != cudaSuccess) return e;
    *used = true;
    return launch_pdl(reinterpret_cast<const void *>(kern), grid, threads,
                      smem, st, p, stages, units, rs, (uint32_t)plane_off);
}

template <int BITS, int MT, int MODE>
static cudaError_t launch_stream_t(const DenseParams &p, cudaStream_t st,
                                   bool *used) {
    // four tokens hold 64 registers of activations: two rows per thread
    return launch_stream_r<BITS, MT, MODE, MT == 4 ? 2 : kRowsPerThread>(
        p, st, used);
}

static bool aligned16(const void *q) {
    return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
}

// Launches the streaming kernel when the shape allows it (M <= 4, row
// strides of scales multiple of 16 bytes, 16-byte aligned bases); *used
// tells the caller whether it ran.
cudaError_t launch_stream(int mode, const DenseParams &p, cudaStream_t st,
                          bool *used) {
    *used = false;
    if (p.M > 4 || (p.G % 8) != 0 || !aligned16(p.sc) || !aligned16(p.bi) ||
        !aligned16(p.wq) || p.group != kGroup)
        return cudaSuccess;
    const int mt = p.M <= 1 ? 1 : p.M <= 2 ? 2 : 4;
    // A plain projection runs as one section: the same kernel as the fused
    // QKV projection, so that a layer's calls share their code.
    DenseParams q = p;
    if (mode == kSPlain) {
        q.nsec = 1;
        q.sec_start[0] = 0;
        q.sec_start[1] = p.N;
        q.sec_out[0] = p.y;
        q.sec_bias[0] = nullptr;
        mode = kSSections;
    }
#define GWA_STREAM_CASE(B, MTV)                                              \
    if (p.bits == B && mt == MTV) {                                          \
        if (mode == kSSections)                                              \
            return launch_stream_t<B, MTV, kSSections>(q, st, used);         \
        if (mode == kSRope)                                                  \
            return launch_stream_t<B, MTV, kSRope>(q, st, used);             \
        return launch_stream_t<B, MTV, kSGateUp>(q, st, used);               \
    }
    GWA_STREAM_CASE(4, 1)
    GWA_STREAM_CASE(4, 2)
    GWA_STREAM_CASE(4, 4)
    GWA_STREAM_CASE(8, 1)
    GWA_STREAM_CASE(8, 2)
    GWA_STREAM_CASE(8, 4)
    GWA_STREAM_CASE(kFp8, 1)
    GWA_STREAM_CASE(kFp8, 2)
    GWA_STREAM_CASE(kFp8, 4)
#undef GWA_STREAM_CASE
    return cudaSuccess;
}

bool stream_eligible(const DenseParams &p) {
    if ((p.G % 8) != 0 || !aligned16(p.sc) || !aligned16(p.bi) ||
        !aligned16(p.wq))
        return false;
    const int nwh = (p.nch + kWarp - 1) / kWarp;
    return nwh * kWarp + kWarp <= kStreamMaxThreads;
}

unsigned int stream_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_stream_timeouts, sizeof v);
    if (reset) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_stream_timeouts, &z, sizeof z);
    }
    return v;
}

}  // namespace gwa
