// Decode (M <= 8) GEMV building blocks: activation staging in shared memory
// and the per-warp row dot products.  Used by the dense kernels (qmv,
// fused sections, gate+up SwiGLU) and by the MoE gather kernels.
//
// Work split: a warp owns a block of R weight rows; its 32 lanes walk the
// 16-byte chunks of those rows (chunk c = lane, lane+32, ...), so each warp
// load instruction moves 512 contiguous bytes per row.  A lane unpacks each
// word once per row and reuses it for every token; it reads the staged
// activations of a chunk once and reuses them for all R rows.  Per chunk the
// lane keeps fp32 pair accumulators, removes the magic constants with the
// precomputed chunk sums and applies the group's scale and bias:
//   y += s * (sum_k x_k f_k - sum_k C_k x_k) + b * sum_k x_k.
// Lanes are reduced with warp shuffles at the end of the row block.
#pragma once

#include "common.cuh"

namespace gwa {

// ------------------------------------------------------------ staging
// Shared-memory image of the activations of `mt` tokens, chunk-major so that
// the 32 lanes of a warp read 32 consecutive 16-byte slots:
//   XF32:  float4 q[m][e][c], e < kChunkCodes/4  (fp32, in unpack order)
//   bf16:  uint4  q[m][e][c], e < kChunkCodes/8  (bf16 pairs, unpack order)
// followed by float2 sums[m][c] = (sum_k C_k x_k, sum_k x_k) per chunk.
template <int BITS, bool XF32>
struct XStage {
    static constexpr int kQuads =
        XF32 ? Fmt<BITS>::kChunkCodes / 4 : Fmt<BITS>::kChunkCodes / 8;
    static __host__ __device__ size_t bytes(int mt, int nch) {
        return (size_t)mt * nch * (16 * kQuads + sizeof(float2));
    }
};

// Stage tokens `tok[0..mt)` (rows of x, K = nch * chunk codes) into shared
// memory; token slots with tok[m] < 0 are zero-filled.  Called by the whole
// CTA; the caller synchronizes afterwards.
template <int BITS, bool XF32>
__device__ __forceinline__ void stage_x(const uint16_t *__restrict__ x,
                                        int64_t x_row_stride,
                                        const int *tok, int mt, int nch,
                                        unsigned char *smem) {
    constexpr int CODES = Fmt<BITS>::kChunkCodes;
    constexpr int Q = XStage<BITS, XF32>::kQuads;
    float2 *sums = reinterpret_cast<float2 *>(
        smem + (size_t)mt * nch * Q * 16);
    const int items = mt * nch;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
        const int m = it / nch, c = it - m * nch;
        float v[CODES];
        if (tok[m] >= 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                x + (int64_t)tok[m] * x_row_stride + (int64_t)c * CODES);
#pragma unroll
            for (int i = 0; i < CODES / 8; ++i) {
                uint4 u = src[i];
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
        // values in unpack order
        float o[CODES];
        float csum = 0.f, xsum = 0.f;
        if constexpr (BITS == 4) {
#pragma unroll
            for (int wd = 0; wd < CODES / 8; ++wd)
#pragma unroll
                for (int i = 0; i < 8; ++i) o[8 * wd + i] = v[8 * wd + u4_perm(i)];
            float odd = 0.f, even = 0.f;
#pragma unroll
            for (int i = 0; i < CODES; i += 2) {
                even += v[i];
                odd += v[i + 1];
            }
            csum = kU4Odd * odd + kU4Even * even;
            xsum = odd + even;
        } else {
#pragma unroll
            for (int i = 0; i < CODES; ++i) {
                o[i] = v[i];
                xsum += v[i];
            }
            csum = kU8Const * xsum;
        }
        if constexpr (XF32) {
            float4 *q = reinterpret_cast<float4 *>(smem);
#pragma unroll
            for (int e = 0; e < Q; ++e)
                q[((size_t)m * Q + e) * nch + c] =
                    make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2],
                                o[4 * e + 3]);
        } else {
            uint4 *q = reinterpret_cast<uint4 *>(smem);
#pragma unroll
            for (int e = 0; e < Q; ++e) {
                uint32_t w4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w4[i] = (uint32_t)f32_to_bf16_bits(o[8 * e + 2 * i]) |
                            ((uint32_t)f32_to_bf16_bits(o[8 * e + 2 * i + 1])
                             << 16);
                q[((size_t)m * Q + e) * nch + c] =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
        sums[(size_t)m * nch + c] = make_float2(csum, xsum);
    }
}

// Pairs of staged activations for word `wd` of chunk `c`, token m.
template <int BITS, bool XF32>
__device__ __forceinline__ void x_pairs(const unsigned char *smem, int m,
                                        int nch, int c, int wd,
                                        float2 (&xp)[BITS == 4 ? 4 : 2]) {
    constexpr int Q = XStage<BITS, XF32>::kQuads;
    if constexpr (XF32) {
        const float4 *q = reinterpret_cast<const float4 *>(smem);
        if constexpr (BITS == 4) {
            float4 a = q[((size_t)m * Q + 2 * wd) * nch + c];
            float4 b = q[((size_t)m * Q + 2 * wd + 1) * nch + c];
            xp[0] = make_float2(a.x, a.y);
            xp[1] = make_float2(a.z, a.w);
            xp[2] = make_float2(b.x, b.y);
            xp[3] = make_float2(b.z, b.w);
        } else {
            float4 a = q[((size_t)m * Q + wd) * nch + c];
            xp[0] = make_float2(a.x, a.y);
            xp[1] = make_float2(a.z, a.w);
        }
    } else {
        const uint4 *q = reinterpret_cast<const uint4 *>(smem);
        if constexpr (BITS == 4) {
            uint4 a = q[((size_t)m * Q + wd) * nch + c];
            xp[0] = make_float2(bf16_lo(a.x), bf16_hi(a.x));
            xp[1] = make_float2(bf16_lo(a.y), bf16_hi(a.y));
            xp[2] = make_float2(bf16_lo(a.z), bf16_hi(a.z));
            xp[3] = make_float2(bf16_lo(a.w), bf16_hi(a.w));
        } else {
            uint4 a = q[((size_t)m * Q + (wd >> 1)) * nch + c];
            uint32_t lo = (wd & 1) ? a.z : a.x, hi = (wd & 1) ? a.w : a.y;
            xp[0] = make_float2(bf16_lo(lo), bf16_hi(lo));
            xp[1] = make_float2(bf16_lo(hi), bf16_hi(hi));
        }
    }
}

template <int BITS, bool XF32>
__device__ __forceinline__ const float2 *x_sums(const unsigned char *smem,
                                                int mt, int nch) {
    return reinterpret_cast<const float2 *>(
        smem + (size_t)mt * nch * XStage<BITS, XF32>::kQuads * 16);
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
// midx[m]); adds the scaled, bias-corrected chunk dot into acc.
template <int BITS, int MT, int R, bool XF32>
__device__ __forceinline__ void chunk_fma(const ChunkRegs<R> &cr, int c,
                                          int nch, const int (&midx)[MT],
                                          const float2 *sums,
                                          const unsigned char *xs,
                                          float (&acc)[R][MT]) {
    constexpr int PAIRS = BITS == 4 ? 4 : 2;
    float2 a2[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) a2[r][m] = make_float2(0.f, 0.f);
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        float2 xp[MT][PAIRS];
#pragma unroll
        for (int m = 0; m < MT; ++m)
            x_pairs<BITS, XF32>(xs, midx[m], nch, c, wd, xp[m]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t word = wd == 0   ? cr.w[r].x
                                  : wd == 1 ? cr.w[r].y
                                  : wd == 2 ? cr.w[r].z
                                            : cr.w[r].w;
            float2 p[PAIRS];
            if constexpr (BITS == 4)
                unpack_u4(word, p);
            else
                unpack_u8(word, p);
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int i = 0; i < PAIRS; ++i)
                    a2[r][m] = __ffma2_rn(p[i], xp[m][i], a2[r][m]);
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float2 cx = sums[(size_t)midx[m] * nch + c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float d = (a2[r][m].x + a2[r][m].y) - cx.x;
            acc[r][m] = fmaf(cr.s[r], d, fmaf(cr.b[r], cx.y, acc[r][m]));
        }
    }
}

// Partial sums of this lane for R rows and MT staged tokens (not reduced).
// L lanes share a row: the lane walks chunks (lane % L), +L, ...
template <int BITS, int MT, int R, bool XF32, int L = kWarp>
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
    const float2 *sums = x_sums<BITS, XF32>(xs, mt_stage, v.nch);
    ChunkRegs<R> cur;
    load_chunk<BITS, R>(v, rows, c, cur);
    while (true) {
        const int cn = c + L;
        const bool more = cn < v.nch;
        ChunkRegs<R> nxt;
        if (more) load_chunk<BITS, R>(v, rows, cn, nxt);
        chunk_fma<BITS, MT, R, XF32>(cur, c, v.nch, midx, sums, xs, acc);
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
