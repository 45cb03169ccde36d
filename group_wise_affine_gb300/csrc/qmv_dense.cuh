// Decode (M <= 8) GEMV building blocks: activation staging in shared memory
// and the per-warp row dot products.  Used by the dense kernels (qmv,
// fused sections, gate+up SwiGLU) and by the MoE gather kernels.
//
// Work split: a warp owns a block of R weight rows; its 32 lanes walk the
// 16-byte chunks of those rows (chunk c = lane, lane+32, ...), so each warp
// load instruction moves 512 contiguous bytes per row.  A lane splits each
// word into code bytes once per row and reuses them for every token; it reads
// the staged activations of a chunk once and reuses them for all R rows.
// Per chunk the lane forms exact integer dots (dp2a) and applies the group's
// scale and bias in fp32 (see common.cuh):
//   y += (s * 2^E) * D + b * sum_k x_k.
// Lanes are reduced with warp shuffles at the end of the row block.
#pragma once

#include "common.cuh"

namespace gwa {

// ------------------------------------------------------------ staging
// Shared-memory image of the activations of `mt` tokens, encoded for the
// integer dot (int16 pairs in dp2a order, see common.cuh), chunk-major so
// that the 32 lanes of a warp read 32 consecutive 16-byte slots:
//   uint4 q[m][e][c], e < kChunkCodes/8
// followed by float2 aux[m][c] = (group scale 2^E, sum of the chunk's x).
// A marked group (common.cuh, "marked groups") holds raw bf16 pairs in the
// same order and a scale of -1.
template <int BITS>
struct XStage {
    static constexpr int kQuads = Fmt<BITS>::kChunkCodes / 8;
    static __host__ __device__ size_t bytes(int mt, int nch) {
        return (size_t)mt * nch * (16 * kQuads + sizeof(float2));
    }
};

// Stage tokens `tok[0..mt)` (rows of x, K = nch * chunk codes) into shared
// memory; token slots with tok[m] < 0 are zero-filled.  One item per
// (token, group of 64).  *mkflag is set to 1 if any group is marked (the
// caller clears it first).  Called by the whole CTA; the caller
// synchronizes.
template <int BITS>
__device__ __forceinline__ void stage_x(const uint16_t *__restrict__ x,
                                        int64_t x_row_stride,
                                        const int *tok, int mt, int nch,
                                        unsigned char *smem, int *mkflag) {
    constexpr int CODES = Fmt<BITS>::kChunkCodes;
    constexpr int CPG = kGroup / CODES;  // chunks per group
    constexpr int Q = XStage<BITS>::kQuads;
    uint4 *q = reinterpret_cast<uint4 *>(smem);
    float2 *aux = reinterpret_cast<float2 *>(smem + (size_t)mt * nch * Q * 16);
    const int G = nch / CPG;
    const int items = mt * G;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
        const int m = it / G, g = it - m * G;
        float v[kGroup];
        if (tok[m] >= 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                x + (int64_t)tok[m] * x_row_stride + (int64_t)g * kGroup);
#pragma unroll
            for (int i = 0; i < kGroup / 8; ++i) {
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
            for (int i = 0; i < kGroup; ++i) v[i] = 0.f;
        }
        int ef = 0;
#pragma unroll
        for (int i = 0; i < kGroup; ++i) ef = max(ef, f32_exp_field(v[i]));
        float f, finv;
        group_scale(ef, f, finv);
        float re = 0.f, ab = 0.f;
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
            re += i16_resid(v[i], finv);
            ab += fabsf(v[i]);
        }
        const bool marked = group_marked(re, ab * finv);
        if (marked) *mkflag = 1;
#pragma unroll
        for (int cg = 0; cg < CPG; ++cg) {
            const int c = g * CPG + cg;
            const float *vc = v + cg * CODES;
            uint32_t pr[CODES / 2];
            float xs = 0.f;
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                if constexpr (BITS == 4) {
                    const float *vw = vc + 8 * wd;
                    uint32_t t[4];
                    u4_pairs(vw, finv, t);
                    if (marked) {  // raw bf16 in the same dp2a order
                        t[0] = raw_pair(vw[0], vw[2]);
                        t[1] = raw_pair(vw[4], vw[6]);
                        t[2] = raw_pair(vw[1], vw[3]);
                        t[3] = raw_pair(vw[5], vw[7]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) pr[4 * wd + i] = t[i];
                } else {
                    const float *vw = vc + 4 * wd;
                    uint32_t t[2];
                    u8_pairs(vw, finv, t);
                    if (marked) {
                        t[0] = raw_pair(vw[0], vw[1]);
                        t[1] = raw_pair(vw[2], vw[3]);
                    }
                    pr[2 * wd] = t[0];
                    pr[2 * wd + 1] = t[1];
                }
            }
#pragma unroll
            for (int i = 0; i < CODES; ++i) xs += vc[i];
#pragma unroll
            for (int e = 0; e < Q; ++e)
                q[((size_t)m * Q + e) * nch + c] =
                    make_uint4(pr[4 * e], pr[4 * e + 1], pr[4 * e + 2],
                               pr[4 * e + 3]);
            aux[(size_t)m * nch + c] = make_float2(marked ? -1.f : f, xs);
        }
    }
}

// Activation pairs of word `wd` of chunk `c`, staged token m.
template <int BITS>
__device__ __forceinline__ void x_pairs(const unsigned char *smem, int m,
                                        int nch, int c, int wd,
                                        uint32_t (&pr)[BITS == 4 ? 4 : 2]) {
    constexpr int Q = XStage<BITS>::kQuads;
    const uint4 *q = reinterpret_cast<const uint4 *>(smem);
    if constexpr (BITS == 4) {
        const uint4 a = q[((size_t)m * Q + wd) * nch + c];
        pr[0] = a.x;
        pr[1] = a.y;
        pr[2] = a.z;
        pr[3] = a.w;
    } else {
        const uint4 a = q[((size_t)m * Q + (wd >> 1)) * nch + c];
        pr[0] = (wd & 1) ? a.z : a.x;
        pr[1] = (wd & 1) ? a.w : a.y;
    }
}

template <int BITS>
__device__ __forceinline__ const float2 *x_aux(const unsigned char *smem,
                                               int mt, int nch) {
    return reinterpret_cast<const float2 *>(
        smem + (size_t)mt * nch * XStage<BITS>::kQuads * 16);
}

// ------------------------------------------------------------ row dots
// Weight view: rows of `nch` 16-byte chunks and G groups.
struct WView {
    const uint4 *wq;
    const uint16_t *sc;
    const uint16_t *bi;
    int nch;
    int G;
};

template <int R>
struct ChunkRegs {
    uint4 w[R];
    float s[R];
    float b[R];
};

template <int BITS, int R>
__device__ __forceinline__ void load_chunk(const WView &v,
                                           const int64_t (&rows)[R], int c,
                                           ChunkRegs<R> &out) {
    constexpr int CODES = Fmt<BITS>::kChunkCodes;
    const int g = (c * CODES) / kGroup;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (rows[r] >= 0) {
            out.w[r] = ld_stream(v.wq + rows[r] * v.nch + c);
            out.s[r] = bf16_bits_to_f32(ld_u16(v.sc + rows[r] * v.G + g));
            out.b[r] = bf16_bits_to_f32(ld_u16(v.bi + rows[r] * v.G + g));
        } else {
            out.w[r] = make_uint4(0, 0, 0, 0);
            out.s[r] = 0.f;
            out.b[r] = 0.f;
        }
    }
}

// One 16-byte chunk of R rows against MT staged tokens (stage slots
// midx[m]); adds the scaled, bias-corrected chunk dot into acc.  With EX
// (some staged group is marked), a marked token's chunk (raw bf16 pairs,
// scale -1) takes the same dot in fp32.
template <int BITS, int MT, int R, bool EX>
__device__ __forceinline__ void chunk_fma(const ChunkRegs<R> &cr, int c,
                                          int nch, const int (&midx)[MT],
                                          const float2 *aux,
                                          const unsigned char *xs,
                                          float (&acc)[R][MT]) {
    constexpr int PAIRS = BITS == 4 ? 4 : 2;
    float2 fa[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) fa[m] = aux[(size_t)midx[m] * nch + c];
    // marked tokens first (raw bf16 pairs, scale -1: fp32 dot one row at a
    // time), so that the integer accumulators below are not live meanwhile
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (!EX || fa[m].x >= 0.f) continue;
        uint32_t xp[4 * PAIRS];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            uint32_t t[PAIRS];
            x_pairs<BITS>(xs, midx[m], nch, c, wd, t);
#pragma unroll
            for (int i = 0; i < PAIRS; ++i) xp[wd * PAIRS + i] = t[i];
        }
#pragma unroll 1
        for (int r = 0; r < R; ++r) {
            const float v = chunk_dot_f32<BITS>(pick(cr.w, r), xp);
            const float sr = pick(cr.s, r), br = pick(cr.b, r);
#pragma unroll
            for (int k = 0; k < R; ++k)
                if (k == r) acc[k][m] = fmaf(sr, v, fmaf(br, fa[m].y, acc[k][m]));
        }
    }
    int d[R][MT][2];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) d[r][m][0] = d[r][m][1] = 0;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        uint32_t xp[MT][PAIRS];
#pragma unroll
        for (int m = 0; m < MT; ++m)
            x_pairs<BITS>(xs, midx[m], nch, c, wd, xp[m]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t word = wd == 0   ? cr.w[r].x
                                  : wd == 1 ? cr.w[r].y
                                  : wd == 2 ? cr.w[r].z
                                            : cr.w[r].w;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if constexpr (BITS == 4)
                    word_dot_u4(word, xp[m], d[r][m]);
                else
                    word_dot_u8(word, xp[m], d[r][m]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (EX && fa[m].x < 0.f) continue;
#pragma unroll
        for (int r = 0; r < R; ++r)
            acc[r][m] = fmaf(cr.s[r] * fa[m].x, (float)dot_total<BITS>(d[r][m]),
                             fmaf(cr.b[r], fa[m].y, acc[r][m]));
    }
}

// Partial sums of this lane for R rows and MT staged tokens (not reduced).
// L lanes share a row: the lane walks chunks (lane % L), +L, ...
template <int BITS, int MT, int R, bool EX, int L = kWarp>
__device__ __forceinline__ void rows_dot(const WView &v,
                                         const int64_t (&rows)[R],
                                         const int (&midx)[MT], int mt_stage,
                                         const unsigned char *xs, int lane,
                                         float (&acc)[R][MT]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
    int c = lane % L;
    if (c >= v.nch) return;
    const float2 *aux = x_aux<BITS>(xs, mt_stage, v.nch);
    ChunkRegs<R> cur;
    load_chunk<BITS, R>(v, rows, c, cur);
    while (true) {
        const int cn = c + L;
        const bool more = cn < v.nch;
        ChunkRegs<R> nxt;
        if (more) load_chunk<BITS, R>(v, rows, cn, nxt);
        chunk_fma<BITS, MT, R, EX>(cur, c, v.nch, midx, aux, xs, acc);
        if (!more) break;
        c = cn;
        cur = nxt;
    }
}

// Sum over the L lanes that share a row (aligned groups of L lanes).
template <int L>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int R, int MT, int L = kWarp>
__device__ __forceinline__ void warp_reduce(float (&acc)[R][MT]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = group_sum<L>(acc[r][m]);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

}  // namespace gwa
