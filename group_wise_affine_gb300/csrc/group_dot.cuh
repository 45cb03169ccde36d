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
    bool mk[MT];          // marked chunk (common.cuh, "marked groups")
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
//   xs[r][g], and for split images xs2[r][g].  The two-plane path later
//   writes each chunk's int8 residual plane over the first half of the
//   pairs (group_plane_store), once every lane holds its pairs in
//   registers.
__host__ __device__ constexpr size_t ximg_bytes(int R, int G,
                                                bool split = false) {
    return (size_t)R * G * (8 * 16 + 8 + (split ? 4 : 0));
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

// Slot (16-byte piece of a chunk's residual plane) that holds quarter q's
// entries in the two-plane path: the pieces follow the order in which
// lds_group loads the chunk's codes (rotation rot = chunk_rot(g)), so
// register piece v of the codes meets plane slots 2v, 2v + 1 (u4) or v (u8).
template <int BITS>
__device__ __forceinline__ int group_lo_slot(int q, int rot) {
    return BITS == 4 ? 2 * (((q >> 1) - rot) & 1) + (q & 1) : (q - rot) & 3;
}

// Four bytes (the low byte of each word) packed into one word, a first.
__device__ __forceinline__ uint32_t pack_bytes(uint32_t a, uint32_t b,
                                               uint32_t c, uint32_t d) {
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040),
                       0x5410);
}

// How an encoder settles a chunk's mark: RAW agrees on it through shuffles
// before forming the pairs and stores a marked chunk's raw bf16 pairs (fp32
// path); DEFER always stores the int16 pairs and adds up the chunk's
// criterion afterwards, off the pairs' path (two-plane path: a marked chunk
// only sets the flag).
enum MarkMode { kMarkRaw = 0, kMarkDefer = 1 };

// Quarter `q` (16 inputs) of group g of image row r, from its 8 packed bf16
// words.  The four quarters of a group sit in four adjacent lanes and agree
// on the group's exponent, sum and mark through shuffles, so every lane of
// the warp must call this.  u4: the high-nibble products of the dot come
// out 16x too large and exact, so f is stored as 2^E / 16.  Marks (common.cuh,
// "marked groups"): with kMarkRaw a marked chunk sets *mkflag (when given)
// to 1 and stores its raw bf16 pairs in the same order and f = -1/16 (u4)
// or -1 (u8), the unit of the fp32 dot; with kMarkDefer the pairs and f are
// always the usual ones and a marked chunk sets *mkflag.  The criterion is
// linear in the quarters' residuals and magnitudes, so each quarter's part
// R_q - 2^-16 A_q is formed alone and the four are added by two shuffles.
template <int BITS, bool SPLIT = false, int MK = kMarkRaw>
__device__ __forceinline__ void encode_quarter(const uint32_t (&u)[8],
                                               bool store, int r, int g, int q,
                                               int R, int G,
                                               unsigned char *img,
                                               int *mkflag = nullptr) {
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
    // rounding error and magnitude of the chunk in units of f
    float re = 0.f, ab = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        re += i16_resid(v[i], finv);
        ab += fabsf(v[i]);
    }
    bool marked = false;
    if constexpr (MK == kMarkRaw) {
        re += __shfl_xor_sync(0xffffffffu, re, 1);
        re += __shfl_xor_sync(0xffffffffu, re, 2);
        ab += __shfl_xor_sync(0xffffffffu, ab, 1);
        ab += __shfl_xor_sync(0xffffffffu, ab, 2);
        marked = group_marked(re, ab * finv);
    }
    auto pair = [&](float a, float b) {
        return marked ? raw_pair(a, b) : i16_pair_fast(a, b, finv);
    };
    uint32_t pr[8];
    if constexpr (BITS == 4) {
        // words 2q, 2q+1: (x0,x2) (x4,x6) (x1,x3) (x5,x7) each
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const float *vw = v + 8 * w;
            pr[4 * w + 0] = pair(vw[0], vw[2]);
            pr[4 * w + 1] = pair(vw[4], vw[6]);
            pr[4 * w + 2] = pair(vw[1], vw[3]);
            pr[4 * w + 3] = pair(vw[5], vw[7]);
        }
    } else {
        // words 4q..4q+3: (x0,x1) (x2,x3) each
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            pr[2 * w] = pair(v[4 * w], v[4 * w + 1]);
            pr[2 * w + 1] = pair(v[4 * w + 2], v[4 * w + 3]);
        }
    }
    if (store) {
        pairs[((size_t)r * 8 + 2 * q) * G + g] =
            make_uint4(pr[0], pr[1], pr[2], pr[3]);
        pairs[((size_t)r * 8 + 2 * q + 1) * G + g] =
            make_uint4(pr[4], pr[5], pr[6], pr[7]);
        if (q == 0) {
            const float unit = BITS == 4 ? 0.0625f : 1.f;
            xf[(size_t)r * G + g] = marked ? -unit : f * unit;
            if (marked && mkflag) *mkflag = 1;
            xsm[(size_t)r * G + g] = sum;
        }
        if (SPLIT && q == 2) xsm[(size_t)R * G + (size_t)r * G + g] = sum;
    }
    if constexpr (MK == kMarkDefer) {
        float d = fmaf(ab * finv, -1.0f / 65536.0f, re);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        if (store && q == 0 && d > 0.f && mkflag) *mkflag = 1;
    }
}


// All `ncons` threads (whole warps) encode R rows of K activations into the
// image: row r from x + src(r) * K, src(r) = rowsrc ? rowsrc[r] : r (rows
// >= Rv encode as zeros); *mkflag, when given, is set to 1 if any group
// is marked (the caller clears it first).  A thread issues
// the loads of up to kXBatch quarters before encoding any, so a long image
// costs about one memory round trip.
constexpr int kXBatch = 4;

template <int BITS, bool SPLIT = false, int MK = kMarkRaw>
__device__ __forceinline__ void encode_rows_shared(
    const uint16_t *__restrict__ x, int Rv, int R, int K, int G, int tid,
    int ncons, unsigned char *img, const int *rowsrc = nullptr,
    int *mkflag = nullptr) {
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
            encode_quarter<BITS, SPLIT, MK>(u[j], it < items, r, rem >> 2,
                                            rem & 3, R, G, img, mkflag);
        }
    }
}

// The int8 residual planes of the two-plane path (common.cuh, "marked
// groups") for an image of R rows: all `ncons` threads take the (row, chunk,
// quarter) items in turn, read the quarter's 16 raw bf16 activations from x
// again (row r from x + src(r) * K, src(r) = rowsrc ? rowsrc[r] : r; the
// encoder's pairs kept only their rounded values), and write its residual
// entries, exact for every chunk, marked or not: slot group_lo_slot(q,
// chunk_rot(g)) of chunk g of row r at lo[(r * 4 + slot) * G + g].  Entries
// in dp4a order: per u4 word those of its low nibbles' inputs (x0 x2 x4 x6),
// then of its high nibbles' (x1 x3 x5 x7); per u8 word x0..x3.  The caller
// brackets this with barriers (the planes may overwrite the image's pairs
// once every lane holds them in registers: lo = the image itself, R = 1).
// Each thread issues the loads of two items before using either (the
// callers' pairs occupy 32 registers meanwhile).
template <int BITS>
__device__ __forceinline__ void group_plane_store(const uint16_t *__restrict__ x,
                                                  int K, int R, int G,
                                                  const int *rowsrc, int tid,
                                                  int ncons,
                                                  const unsigned char *img,
                                                  uint4 *lo) {
    const float *xf = reinterpret_cast<const float *>(
        reinterpret_cast<const uint4 *>(img) + (size_t)R * 8 * G);
    const int items = R * 4 * G;
    constexpr int B = 2;
    for (int b0 = tid; b0 < items; b0 += B * ncons) {
        uint4 u[B][2];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int it = b0 + j * ncons;
            if (it < items) {
                const int r = it / (4 * G), rem = it - r * 4 * G;
                const int sr = rowsrc ? rowsrc[r] : r;
                const uint4 *src = reinterpret_cast<const uint4 *>(
                                       x + (int64_t)sr * K) + 2 * rem;
                u[j][0] = src[0];
                u[j][1] = src[1];
            }
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int it = b0 + j * ncons;
            if (it >= items) break;
            const int r = it / (4 * G), rem = it - r * 4 * G;
            const int g = rem >> 2, q = rem & 3;
            // the pairs' unit: f as stored (u4: 2^E / 16), so 2^-E is
            const float fs = fabsf(xf[(size_t)r * G + g]);
            const float finv = 1.0f / (BITS == 4 ? 16.0f * fs : fs);
            uint32_t w4[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t wv[4] = {u[j][h].x, u[j][h].y, u[j][h].z, u[j][h].w};
                uint32_t e[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    e[2 * k] = i8_resid(bf16_lo(wv[k]), finv);
                    e[2 * k + 1] = i8_resid(bf16_hi(wv[k]), finv);
                }
                if constexpr (BITS == 4) {  // one u4 word: even, then odd
                    w4[2 * h] = pack_bytes(e[0], e[2], e[4], e[6]);
                    w4[2 * h + 1] = pack_bytes(e[1], e[3], e[5], e[7]);
                } else {  // two u8 words
                    w4[2 * h] = pack_bytes(e[0], e[1], e[2], e[3]);
                    w4[2 * h + 1] = pack_bytes(e[4], e[5], e[6], e[7]);
                }
            }
            lo[((size_t)r * 4 + group_lo_slot<BITS>(q, chunk_rot<BITS>(g))) * G + g] =
                make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
    }
}

// A row's group of codes, in chunk_rot order.
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
        const float fm = active ? xf[(size_t)r * G + g] : 0.f;
        gx.mk[m] = fm < 0.f;  // raw-marked images (kMarkRaw)
        gx.f[m] = fabsf(fm);
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

// Plane entries of word c of register piece v (two words per u4 word, one
// per u8 word), from the piece's plane slots as loaded: u4 slots 2v, 2v + 1
// in e0, e1 (word c in e[c / 2], halves c % 2); u8 slot v in e0.
template <int BITS>
__device__ __forceinline__ uint2 plane_words(const uint4 &e0, const uint4 &e1,
                                             int c) {
    if constexpr (BITS == 4) {
        const uint4 &e = c < 2 ? e0 : e1;
        return (c & 1) ? make_uint2(e.z, e.w) : make_uint2(e.x, e.y);
    } else {
        return make_uint2(c == 0 ? e0.x : c == 1 ? e0.y : c == 2 ? e0.z : e0.w,
                          0u);
    }
}

// group_dot and the residual-plane dot of the two-plane path in one pass
// over the code bytes: dh as group_dot's d; dl the same dot with the plane
// at lo[0], lo[stride], ... (slots as group_lo_slot), read a 16-byte slot
// at a time, its scale 2^-7 of dh's.  w as lds_group loaded it.
template <int BITS, int MT>
__device__ __forceinline__ void group_dot2(const uint4 (&w)[BITS / 2],
                                           const GroupX<MT> &gx, const uint4 *lo,
                                           int stride, int (&dh)[MT], int &dl) {
    constexpr int NV = BITS / 2;
    int a[MT][4], b[2] = {0, 0};
#pragma unroll
    for (int m = 0; m < MT; ++m) a[m][0] = a[m][1] = a[m][2] = a[m][3] = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const uint4 e0 = lo[(size_t)(BITS == 4 ? 2 * v : v) * stride];
        const uint4 e1 = BITS == 4 ? lo[(size_t)(2 * v + 1) * stride] : e0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int wd = 4 * v + c;
            const uint32_t word = c == 0 ? w[v].x : c == 1 ? w[v].y
                                  : c == 2 ? w[v].z : w[v].w;
            const uint2 e = plane_words<BITS>(e0, e1, c);
            if constexpr (BITS == 4) {
                const uint32_t l = word & 0x0f0f0f0fu;
                const uint32_t h = word & 0xf0f0f0f0u;
                const int p = (wd & 1) * 2;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = gx.pr[m] + 4 * wd;
                    a[m][p] = dp2a_hi(pr[1], l, dp2a_lo(pr[0], l, a[m][p]));
                    a[m][p + 1] = dp2a_hi(pr[3], h, dp2a_lo(pr[2], h, a[m][p + 1]));
                }
                b[0] = dp4a_us(l, e.x, b[0]);
                b[1] = dp4a_us(h, e.y, b[1]);
            } else {
                const int p = wd & 3;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = gx.pr[m] + 2 * wd;
                    a[m][p] = dp2a_hi(pr[1], word, dp2a_lo(pr[0], word, a[m][p]));
                }
                b[wd & 1] = dp4a_us(word, e.x, b[wd & 1]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
        dh[m] = BITS == 4 ? 16 * (a[m][0] + a[m][2]) + (a[m][1] + a[m][3])
                          : (a[m][0] + a[m][1]) + (a[m][2] + a[m][3]);
    dl = BITS == 4 ? 16 * b[0] + b[1] : b[0] + b[1];
}

// The residual-plane dot of group_dot_split's halves: dl over inputs
// [0, 32), dh over [32, 64), scaled like group_dot2's dl (slots as
// group_lo_slot; rot decides which half a register piece falls in).
template <int BITS>
__device__ __forceinline__ void group_dot_lo_split(const uint4 (&w)[BITS / 2],
                                                   const uint4 *lo, int stride,
                                                   int rot, int &dl, int &dh) {
    constexpr int NV = BITS / 2;
    dl = dh = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int pc = (v + rot) & (NV - 1);
        const uint4 e0 = lo[(size_t)(BITS == 4 ? 2 * v : v) * stride];
        const uint4 e1 = BITS == 4 ? lo[(size_t)(2 * v + 1) * stride] : e0;
        int b0 = 0, b1 = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t word = c == 0 ? w[v].x : c == 1 ? w[v].y
                                  : c == 2 ? w[v].z : w[v].w;
            const uint2 e = plane_words<BITS>(e0, e1, c);
            if constexpr (BITS == 4) {
                b0 = dp4a_us(word & 0x0f0f0f0fu, e.x, b0);
                b1 = dp4a_us(word & 0xf0f0f0f0u, e.y, b1);
            } else {
                b0 = dp4a_us(word, e.x, b0);
            }
        }
        const int dv = BITS == 4 ? 16 * b0 + b1 : b0;
        if (pc < NV / 2)
            dl += dv;
        else
            dh += dv;
    }
}

// group_dot of token m of a marked chunk, in fp32 (common.cuh): the same
// pairs hold raw bf16 activations and the same code bytes multiply them, so
// the result has group_dot's scale (u4: 16 times the true sum).
// Two fp32 products per instruction (FFMA2): a pair of raw bf16
// activations times a pair of code bytes (bytes i, i + 1 of b, each exact as
// 2^23 + byte - 2^23), into the two lanes of a float2 accumulator.
template <int I>
__device__ __forceinline__ float2 byte_pair_f32(uint32_t b) {
    const float2 t = make_float2(__uint_as_float(__byte_perm(b, 0x4b000000u, 0x7440 | I)),
                                 __uint_as_float(__byte_perm(b, 0x4b000000u, 0x7440 | (I + 1))));
    return __fadd2_rn(t, make_float2(-8388608.0f, -8388608.0f));
}
__device__ __forceinline__ float2 bf16_pair_f32(uint32_t a) {
    return make_float2(bf16_lo(a), bf16_hi(a));
}

template <int BITS, int MT>
__device__ __forceinline__ float group_dot_f32(const uint4 (&w)[BITS / 2],
                                               const GroupX<MT> &gx, int m) {
    // u4: lanes of a0 sum the low nibbles' products, a1 the high ones'
    // (16 q); u8: a0 bytes 0-1, a1 bytes 2-3 of each word
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int v = 0; v < BITS / 2; ++v) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int wd = 4 * v + c;
            const uint32_t word = c == 0 ? w[v].x : c == 1 ? w[v].y
                                  : c == 2 ? w[v].z : w[v].w;
            if constexpr (BITS == 4) {
                const uint32_t *pr = gx.pr[m] + 4 * wd;
                const uint32_t lo = word & 0x0f0f0f0fu, hi = word & 0xf0f0f0f0u;
                a0 = __ffma2_rn(bf16_pair_f32(pr[0]), byte_pair_f32<0>(lo), a0);
                a0 = __ffma2_rn(bf16_pair_f32(pr[1]), byte_pair_f32<2>(lo), a0);
                a1 = __ffma2_rn(bf16_pair_f32(pr[2]), byte_pair_f32<0>(hi), a1);
                a1 = __ffma2_rn(bf16_pair_f32(pr[3]), byte_pair_f32<2>(hi), a1);
            } else {
                const uint32_t *pr = gx.pr[m] + 2 * wd;
                a0 = __ffma2_rn(bf16_pair_f32(pr[0]), byte_pair_f32<0>(word), a0);
                a1 = __ffma2_rn(bf16_pair_f32(pr[1]), byte_pair_f32<2>(word), a1);
            }
        }
    }
    const float s0 = a0.x + a0.y, s1 = a1.x + a1.y;
    return BITS == 4 ? fmaf(s0, 16.f, s1) : s0 + s1;
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
