// Group-per-lane integer dot shared by the one-token decode kernel
// (qmv_group.cu) and the streaming MoE kernels (moe_stream.cu).
//
// A lane owns one chunk of 64 inputs (one quantization group of 64, half a
// group of 128, or two groups of 32).  The activations of that chunk are
// encoded once per CTA into a shared-memory image (int16 pairs with one
// power-of-two scale per chunk, see common.cuh) and then held in 32
// registers per activation row; per weight row the lane forms the exact
// integer dot of its chunk with dp2a and applies the affine map once per
// group it covers:
//   y += (s * 2^E) * D + b * sum_k x_k,   D = sum_k q_k * xi_k,
// with D and sum_k x_k taken over the chunk, or over each half of it for
// groups of 32 ("split" images carry the two half sums).
// Packed format: "saragossa", "Quantization formats" (MLX affine, codes
// lowest bits first, one bf16 scale and bias per 64 inputs).
#pragma once

#include "common.cuh"

namespace gwa {

// Activations of one chunk for MT activation rows, encoded for the dot.
template <int MT>
struct GroupX {
    uint32_t pr[MT][32];  // int16 pairs in dp2a order
    float f[MT];          // 2^E (u4: 2^E / 16, see encode_quarter)
    float xs[MT];         // plain fp32 sum of the chunk's activations
                          // (split: of its first 32)
    float xs2[MT];        // split: plain fp32 sum of its last 32
};

// int16 of v * finv, rounded to nearest even: adding 1.5 * 2^23 puts the
// rounded integer in the low mantissa bits (|v * finv| < 2^15, and the
// product is exact because finv is a power of two).
__device__ __forceinline__ uint32_t i16_bits(float v, float finv) {
    return __float_as_uint(fmaf(v, finv, 12582912.0f));
}
__device__ __forceinline__ uint32_t i16_pair_fast(float a, float b,
                                                  float finv) {
    return __byte_perm(i16_bits(a, finv), i16_bits(b, finv), 0x5410);
}

// Shared-memory image of R encoded activation rows of G chunks, chunk-major
// so that the lanes of a warp (consecutive chunks) read consecutive 16-byte
// pieces:
//   pairs[r][c][g] (uint4: pairs 4c..4c+3 of chunk g), then f[r][g],
//   xs[r][g], and for split images xs2[r][g].
__host__ __device__ constexpr size_t ximg_bytes(int R, int G,
                                                bool split = false) {
    return (size_t)R * G * (8 * 16 + 8 + (split ? 4 : 0));
}

// Quarter `q` (16 inputs) of group g of image row r, from its 8 packed bf16
// words.  The four quarters of a group sit in four adjacent lanes and agree
// on the group's exponent and sum through shuffles, so every lane of the
// warp must call this.  u4: the high-nibble products of the dot come out
// 16x too large and exact, so f is stored as 2^E / 16.
template <int BITS, bool SPLIT = false>
__device__ __forceinline__ void encode_quarter(const uint32_t (&u)[8],
                                               bool store, int r, int g, int q,
                                               int R, int G,
                                               unsigned char *img) {
    uint4 *pairs = reinterpret_cast<uint4 *>(img);
    float *xf = reinterpret_cast<float *>(pairs + (size_t)R * 8 * G);
    float *xsm = xf + (size_t)R * G;
    // largest magnitude (bf16 bits without sign, two per word)
    uint32_t mx = 0u;
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        mx = __vmaxu2(mx, u[i] & 0x7fff7fffu);
        v[2 * i] = bf16_lo(u[i]);
        v[2 * i + 1] = bf16_hi(u[i]);
    }
    uint32_t m16 = max(mx & 0xffffu, mx >> 16);
    m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, 1));
    m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, 2));
    float t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = (v[i] + v[i + 4]) + (v[i + 8] + v[i + 12]);
    float sum = (t[0] + t[1]) + (t[2] + t[3]);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);  // quarters 0+1, 2+3
    if constexpr (!SPLIT) sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    float f, finv;
    group_scale((int)((m16 >> 7) & 0xffu), f, finv);
    uint32_t pr[8];
    if constexpr (BITS == 4) {
        // words 2q, 2q+1: (x0,x2) (x4,x6) (x1,x3) (x5,x7) each
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const float *vw = v + 8 * w;
            pr[4 * w + 0] = i16_pair_fast(vw[0], vw[2], finv);
            pr[4 * w + 1] = i16_pair_fast(vw[4], vw[6], finv);
            pr[4 * w + 2] = i16_pair_fast(vw[1], vw[3], finv);
            pr[4 * w + 3] = i16_pair_fast(vw[5], vw[7], finv);
        }
    } else {
        // words 4q..4q+3: (x0,x1) (x2,x3) each
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            pr[2 * w] = i16_pair_fast(v[4 * w], v[4 * w + 1], finv);
            pr[2 * w + 1] = i16_pair_fast(v[4 * w + 2], v[4 * w + 3], finv);
        }
    }
    if (store) {
        pairs[((size_t)r * 8 + 2 * q) * G + g] =
            make_uint4(pr[0], pr[1], pr[2], pr[3]);
        pairs[((size_t)r * 8 + 2 * q + 1) * G + g] =
            make_uint4(pr[4], pr[5], pr[6], pr[7]);
        if (q == 0) {
            xf[(size_t)r * G + g] = BITS == 4 ? f * 0.0625f : f;
            xsm[(size_t)r * G + g] = sum;
        }
        if (SPLIT && q == 2) xsm[(size_t)R * G + (size_t)r * G + g] = sum;
    }
}

// All `ncons` threads (whole warps) encode R rows of K activations into the
// image: row r from x + src(r) * K, src(r) = rowsrc ? rowsrc[r] : r (rows
// >= Rv encode as zeros).  A thread issues
// the loads of up to kXBatch quarters before encoding any, so a long image
// costs about one memory round trip.
constexpr int kXBatch = 4;

template <int BITS, bool SPLIT = false>
__device__ __forceinline__ void encode_rows_shared(
    const uint16_t *__restrict__ x, int Rv, int R, int K, int G, int tid,
    int ncons, unsigned char *img, const int *rowsrc = nullptr) {
    const int items = R * G * 4;
    const int iters = (items + ncons - 1) / ncons;  // same for every thread
    for (int b0 = 0; b0 < iters; b0 += kXBatch) {
        uint32_t u[kXBatch][8];
#pragma unroll
        for (int j = 0; j < kXBatch; ++j) {
            const int it = (b0 + j) * ncons + tid;
            const int r = it / (4 * G);
            if (b0 + j < iters && it < items && r < Rv) {
                const int rem = it - r * 4 * G;
                const int sr = rowsrc ? rowsrc[r] : r;
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    x + (int64_t)sr * K + (int64_t)(rem >> 2) * kGroup +
                    (rem & 3) * 16);
                const uint4 a = src[0], b = src[1];
                u[j][0] = a.x; u[j][1] = a.y; u[j][2] = a.z; u[j][3] = a.w;
                u[j][4] = b.x; u[j][5] = b.y; u[j][6] = b.z; u[j][7] = b.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) u[j][i] = 0u;
            }
        }
#pragma unroll
        for (int j = 0; j < kXBatch; ++j) {
            if (b0 + j >= iters) break;  // uniform: the shuffles need every lane
            const int it = (b0 + j) * ncons + tid;
            const int r = it / (4 * G), rem = it - r * 4 * G;
            encode_quarter<BITS, SPLIT>(u[j], it < items, r, rem >> 2, rem & 3,
                                        R, G, img);
        }
    }
}

// Bank-conflict-free reads of a row's group.  Lane g reads its group's
// 16-byte code chunks starting at chunk rot(g), so the lanes whose groups
// lie 128 bytes apart (4 apart for u4, 2 apart for u8) read different banks
// in the same instruction.  Its activation pairs are loaded in the same
// rotated order (image chunk shift), so the dot is unchanged.
template <int BITS>
__device__ __forceinline__ int chunk_rot(int g) {
    return BITS == 4 ? (g >> 2) & 1 : (g >> 1) & 3;
}
template <int BITS>
__device__ __forceinline__ int image_shift(int g) {
    return (BITS == 4 ? 4 : 2) * chunk_rot<BITS>(g);
}
template <int BITS>
__device__ __forceinline__ void lds_group(const unsigned char *src, int rot,
                                          uint4 (&w)[BITS / 2]) {
    constexpr int NV = BITS / 2;
#pragma unroll
    for (int i = 0; i < NV; ++i)
        w[i] = reinterpret_cast<const uint4 *>(src)[(i + rot) & (NV - 1)];
}

// Image rows r0 .. r0+MT-1 of group g into registers (zeros when !active),
// image chunks rotated by `shift` (see chunk_rot).
template <int MT, bool SPLIT = false>
__device__ __forceinline__ void load_group_rows(const unsigned char *img,
                                                int R, int G, int r0, int g,
                                                bool active, GroupX<MT> &gx,
                                                int shift = 0) {
    const uint4 *pairs = reinterpret_cast<const uint4 *>(img);
    const float *xf = reinterpret_cast<const float *>(pairs + (size_t)R * 8 * G);
    const float *xsm = xf + (size_t)R * G;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int r = r0 + m;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 t = pairs[((size_t)r * 8 + ((c + shift) & 7)) * G + g];
            gx.pr[m][4 * c] = t.x;
            gx.pr[m][4 * c + 1] = t.y;
            gx.pr[m][4 * c + 2] = t.z;
            gx.pr[m][4 * c + 3] = t.w;
        }
        gx.f[m] = active ? xf[(size_t)r * G + g] : 0.f;
        gx.xs[m] = active ? xsm[(size_t)r * G + g] : 0.f;
        gx.xs2[m] = SPLIT && active ? xsm[(size_t)R * G + (size_t)r * G + g] : 0.f;
    }
}

// Exact integer dot of one row's group (BITS*2 words) with the encoded
// activations; four accumulators per token keep the dp2a chains short.
// Returns D16 = 16 * D_lo + D_hi (u4) or D (u8).
template <int BITS, int MT>
__device__ __forceinline__ void group_dot(const uint4 (&w)[BITS / 2],
                                          const GroupX<MT> &gx,
                                          int (&d)[MT]) {
    int a[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m) a[m][0] = a[m][1] = a[m][2] = a[m][3] = 0;
#pragma unroll
    for (int v = 0; v < BITS / 2; ++v) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int wd = 4 * v + c;
            const uint32_t word = c == 0 ? w[v].x : c == 1 ? w[v].y
                                  : c == 2 ? w[v].z : w[v].w;
            if constexpr (BITS == 4) {
                const uint32_t lo = word & 0x0f0f0f0fu;
                const uint32_t hi = word & 0xf0f0f0f0u;
                const int p = (wd & 1) * 2;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = gx.pr[m] + 4 * wd;
                    a[m][p] = dp2a_hi(pr[1], lo, dp2a_lo(pr[0], lo, a[m][p]));
                    a[m][p + 1] =
                        dp2a_hi(pr[3], hi, dp2a_lo(pr[2], hi, a[m][p + 1]));
                }
            } else {
                const int p = wd & 3;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = gx.pr[m] + 2 * wd;
                    a[m][p] = dp2a_hi(pr[1], word, dp2a_lo(pr[0], word, a[m][p]));
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if constexpr (BITS == 4)
            d[m] = 16 * (a[m][0] + a[m][2]) + (a[m][1] + a[m][3]);
        else
            d[m] = (a[m][0] + a[m][1]) + (a[m][2] + a[m][3]);
    }
}

// The same dot split over the chunk's two halves (groups of 32): dl over
// inputs [0, 32), dh over [32, 64), each scaled like group_dot's result.
// Register piece v of w holds code piece (v + rot) & (NV - 1) (lds_group
// with rotation rot), so which half a piece falls in is known only at run
// time: each piece keeps its own sums and they are assigned at the end.
template <int BITS, int MT>
__device__ __forceinline__ void group_dot_split(const uint4 (&w)[BITS / 2],
                                                const GroupX<MT> &gx, int rot,
                                                int (&dl)[MT], int (&dh)[MT]) {
    constexpr int NV = BITS / 2;
    int a[NV][MT][2];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int m = 0; m < MT; ++m) a[v][m][0] = a[v][m][1] = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int wd = 4 * v + c;
            const uint32_t word = c == 0 ? w[v].x : c == 1 ? w[v].y
                                  : c == 2 ? w[v].z : w[v].w;
            if constexpr (BITS == 4) {
                const uint32_t lo = word & 0x0f0f0f0fu;
                const uint32_t hi = word & 0xf0f0f0f0u;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = gx.pr[m] + 4 * wd;
                    a[v][m][0] = dp2a_hi(pr[1], lo, dp2a_lo(pr[0], lo, a[v][m][0]));
                    a[v][m][1] = dp2a_hi(pr[3], hi, dp2a_lo(pr[2], hi, a[v][m][1]));
                }
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = gx.pr[m] + 2 * wd;
                    a[v][m][c & 1] =
                        dp2a_hi(pr[1], word, dp2a_lo(pr[0], word, a[v][m][c & 1]));
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        int lo = 0, hi = 0;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int dv = BITS == 4 ? 16 * a[v][m][0] + a[v][m][1]
                                     : a[v][m][0] + a[v][m][1];
            if (((v + rot) & (NV - 1)) < NV / 2)
                lo += dv;
            else
                hi += dv;
        }
        dl[m] = lo;
        dh[m] = hi;
    }
}

// Transpose reduction of V values across aligned groups of W lanes (W a
// power of two, 2..32; the W-lane groups of a warp reduce independently).
// Afterwards lane l of a group holds the group sum of value index
// l >> (log2 W - log2 V); lanes whose low (log2 W - log2 V) bits are zero
// hold each index once.  Every lane of the warp must call this.
template <int W, int V>
__device__ __forceinline__ float sub_reduce(float (&v)[V], int lane) {
    static_assert(W >= 2 && W <= 32 && (W & (W - 1)) == 0, "W");
    static_assert(V >= 1 && V <= W && (V & (V - 1)) == 0, "V");
#pragma unroll
    for (int half = V / 2, bit = W / 2; half >= 1; half /= 2, bit /= 2) {
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const bool up = (lane & bit) != 0;
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    float r = v[0];
#pragma unroll
    for (int bit = W / (2 * V); bit >= 1; bit /= 2)
        r += __shfl_xor_sync(0xffffffffu, r, bit);
    return r;
}

}  // namespace gwa
