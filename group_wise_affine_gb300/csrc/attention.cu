// Softmax attention over a 4-bit (or 8-bit) value cache with the values
// dequantized inline ("Sanctum-MLX", six-changes table row 5, "Fused
// attention with inline V dequant (sdpa_dequant_v)", and the paragraph after
// it: Q, a materialized bf16 K and the compressed V state in; online softmax
// in fp32; causal mask; GQA without copying K or V).  The value format is
// this library's affine one along the head dimension (codes packed 32/b per
// word, lowest bits first; one bf16 scale and bias per 64 dimensions;
// v = scale * code + bias).
//
// Split-K decode (flash-decoding): the keys of each (batch, KV head) are cut
// into splits, one block per split and per group of up to 8 query rows of
// that KV head (its GQA query heads x query positions), so K and V stream
// from HBM once per KV head.  Each warp of a block takes tiles of 16 keys
// and runs both products on the tensor cores with warp-level bf16 MMAs
// (m16n8k16, fp32 accumulation):
//
//   scores  S^T = K Q^T      m = the tile's 16 keys, n = the 8 query rows,
//                            k = the head dimension;
//   values  O^T += C^T P'^T  m = 16 dimensions, n = the query rows,
//                            k = the tile's keys,
//
// where C holds the raw codes (exact small integers in bf16) and P' = P *
// scale of the key's group, so the dequantization folds into the weights:
// sum_t p_t (s_t q_t + b_t) = sum_t (p_t s_t) q_t + sum_t p_t b_t, the bias
// term kept per row and group in fp32.  The online softmax (base 2, scores
// pre-multiplied by log2 e) runs on the scores' accumulator fragments; one
// movmatrix transpose turns them into the value product's operand.  The
// warp's tiles stream through a ring of shared-memory stages filled with
// cp.async several tiles ahead, each lane copying exactly the fragments it
// will read, so no stage needs a barrier.  The warps merge in shared memory
// and the block writes (output, max, sum) per row and split to the
// workspace; a second kernel rescales and adds the splits and writes bf16.
//
// Tensor-core use is small (5-8 live query rows against m16n8k16 tiles);
// the kernel is bound by the K and V bytes it streams, so the warp-level
// MMA, whose fragments live in registers next to the softmax and the code
// unpacking, serves better here than a TMEM-accumulated tcgen05 MMA, whose
// smallest tile is 64 rows.
#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace gwa {

constexpr int kAttRows = 8;    // query rows per block: the MMAs' n
constexpr int kAttWarps = 4;
constexpr int kAttTile = 16;   // keys per warp tile: the MMAs' m / k
constexpr int kAttMaxSplits = 1024;

struct AttParams {
    const uint16_t *q;    // [B, Hq, Lq, D]
    const uint16_t *k;    // [B, Hkv, T, D]
    const uint32_t *vq;   // [B, Hkv, T, D*bits/32]
    const uint16_t *vs;   // [B, Hkv, T, D/64]
    const uint16_t *vb;
    uint16_t *out;        // [B, Hq, Lq, D]
    float *part;          // [B, Hq, Lq, nsplit, D + 2]
    int B, Hq, Hkv, Lq, T, nsplit, rowgroups;
    float scale;
    int causal;
};

// Whether `blocks` blocks of kAttWarps warps with `stages` stages of
// `stage` bytes fit in an SM's 228 KB (2 KB per block for the static
// buffers and the system's share).
constexpr bool att_fits(int stage, int blocks, int stages) {
    return blocks * (kAttWarps * stages * stage + 2048) <= 228 * 1024;
}

// One warp's stage of the ring, in bytes.  Every item is laid out
// [item][lane] so a warp's copies and reads of one item are consecutive.
template <int BITS, int D>
struct AttLayout {
    static constexpr int G = D / 64;          // scale groups per key row
    static constexpr int KC = D / 32;         // 16-byte K chunks per lane and key
    static constexpr int VB = BITS;           // code bytes per lane, key, group
    static constexpr int SB = G >= 2 ? 2 * G : 4;  // scale bytes per lane, key
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + 2 * KC * 16 * kWarp;
    static constexpr int S_OFF = V_OFF + 4 * G * VB * kWarp;
    static constexpr int B_OFF = S_OFF + 2 * SB * kWarp;
    static constexpr int STAGE = B_OFF + 2 * SB * kWarp;
    // stages and resident blocks: three blocks of three stages where they
    // fit in an SM's shared memory, else two blocks of four, three or two
    static constexpr int S = att_fits(STAGE, 3, 3)   ? 3
                             : att_fits(STAGE, 2, 4) ? 4
                             : att_fits(STAGE, 2, 3) ? 3
                                                     : 2;
    static constexpr int BLOCKS_PER_SM = att_fits(STAGE, 3, 3) ? 3 : 2;
    static constexpr int WARP_BYTES = STAGE * S;
    static constexpr int BYTES = WARP_BYTES * kAttWarps;
    static_assert(kAttRows * D * 4 <= WARP_BYTES, "merge buffer fits the ring");
    static_assert(att_fits(STAGE, BLOCKS_PER_SM, S), "shared memory per SM");
};

template <int N>
__device__ __forceinline__ void cp_async(void *dst, const void *src) {
    if constexpr (N == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                     "l"(src)
                     : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(dst)),
                     "l"(src), "n"(N)
                     : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// d += a b on bf16 m16n8k16 fragments (fp32 accumulators).
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The transpose of an 8x8 bf16 matrix held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 pair (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) {
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ __nv_bfloat162 bits_bf2(uint32_t v) {
    return *reinterpret_cast<const __nv_bfloat162 *>(&v);
}

// The 4-bit fields at bits 0-3 and 16-19 of x as an exact bf16 pair:
// 0x4300 | q is 128 + q, and subtracting 128 leaves q.
__device__ __forceinline__ uint32_t codes_bf16x2(uint32_t x) {
    return bf2_bits(__hsub2(bits_bf2((x & 0x000f000fu) | 0x43004300u),
                            bits_bf2(0x43004300u)));
}

template <int BITS, int D>
__global__ void __launch_bounds__(kAttWarps * kWarp,
                                  AttLayout<BITS, D>::BLOCKS_PER_SM)
    attn_partial_kernel(AttParams p) {
    using L = AttLayout<BITS, D>;
    constexpr int G = L::G, KC = L::KC, S = L::S, VB = L::VB, SB = L::SB;
    constexpr int WPR = D * BITS / 32;  // code words per key row
    constexpr int NT = D / 16;          // value m-tiles: four per group
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char att_smem[];
    __shared__ float s_m[kAttWarps][kAttRows], s_l[kAttWarps][kAttRows];
    __shared__ float s_b[kAttWarps][kAttRows][G];

    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x / kWarp;
    const int g = lane >> 2, t = lane & 3;  // fragment row group, column pair
    const int split = blockIdx.x;
    const int hk = blockIdx.y / p.rowgroups, rg = blockIdx.y % p.rowgroups;
    const int b = blockIdx.z;
    const int rep = p.Hq / p.Hkv;
    const int nlive = min(kAttRows, rep * p.Lq - rg * kAttRows);
    const int t0 = (int)((int64_t)p.T * split / p.nsplit);
    const int t1 = (int)((int64_t)p.T * (split + 1) / p.nsplit);
    const int64_t kv = ((int64_t)b * p.Hkv + hk) * p.T;  // first key row
    const int64_t rows_total = (int64_t)p.B * p.Hkv * p.T;
    unsigned char *wsm = att_smem + warp * L::WARP_BYTES;
    if (threadIdx.x == 0) pdl_launch_dependents();
    pdl_wait_primary();  // q, k, v may come from the previous kernel

    // keys [0, tm) are visible to this lane's output rows 2t and 2t + 1
    int tm[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = 2 * t + h;
        const int lq = (rg * kAttRows + r) % p.Lq;
        tm[h] = r >= nlive ? 0 : p.causal ? p.T - p.Lq + lq + 1 : p.T;
    }
    // query row g, chunks 4c + t: the scores' B fragments.  Chunk 4c + t of
    // a row holds dimensions 8(4c + t) .. +7; the k order of the MMA is
    // permuted so that each chunk feeds two k-steps (the same permutation
    // for K).
    uint4 qf[KC];
    if (g < nlive) {
        const int r = rg * kAttRows + g;
        const int hq = hk * rep + r / p.Lq, lq = r % p.Lq;
        const uint4 *qr = reinterpret_cast<const uint4 *>(
            p.q + (((int64_t)b * p.Hq + hq) * p.Lq + lq) * D);
#pragma unroll
        for (int c = 0; c < KC; ++c) qf[c] = qr[4 * c + t];
    } else {
#pragma unroll
        for (int c = 0; c < KC; ++c) qf[c] = make_uint4(0u, 0u, 0u, 0u);
    }

    const int ntile = t1 > t0 ? (t1 - t0 + kAttTile - 1) / kAttTile : 0;
    const int nmine = ntile > warp ? (ntile - warp + kAttWarps - 1) / kAttWarps : 0;
    // Tile i of this warp: keys ts .. ts + 15.  The scores' row g is key
    // 2g and row g + 8 key 2g + 1 (the lane copies those two K rows and
    // their scales and biases); the value product's k = 2t, 2t + 1 are keys
    // 4t, 4t + 2 and k = 2t + 8, 2t + 9 keys 4t + 1, 4t + 3 (the lane copies
    // its 8 dimensions of each group of those four keys).  Keys past the
    // split are clamped to its last key and masked.
    auto issue = [&](int i) {
        unsigned char *st = wsm + (i % S) * L::STAGE;
        const int ts = t0 + (warp + i * kAttWarps) * kAttTile;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int64_t row = kv + min(ts + 2 * g + kk, t1 - 1);
            const uint16_t *src = p.k + row * D + 8 * t;
#pragma unroll
            for (int c = 0; c < KC; ++c)
                cp_async<16>(st + L::K_OFF + ((kk * KC + c) * kWarp + lane) * 16,
                             src + 32 * c);
            unsigned char *ds = st + L::S_OFF + (kk * kWarp + lane) * SB;
            unsigned char *db = st + L::B_OFF + (kk * kWarp + lane) * SB;
            if constexpr (G >= 2) {
                cp_async<SB>(ds, p.vs + row * G);
                cp_async<SB>(db, p.vb + row * G);
            } else if ((row | 1) < rows_total) {
                // one group: the aligned 4-byte window holding the key's entry
                cp_async<4>(ds, p.vs + (row & ~(int64_t)1));
                cp_async<4>(db, p.vb + (row & ~(int64_t)1));
            } else {  // the arrays' last entry, at an even index
                *reinterpret_cast<uint32_t *>(ds) = p.vs[row];
                *reinterpret_cast<uint32_t *>(db) = p.vb[row];
            }
        }
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
            const int64_t row = kv + min(ts + 4 * t + kq, t1 - 1);
            const unsigned char *src =
                reinterpret_cast<const unsigned char *>(p.vq + row * WPR) + g * VB;
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                cp_async<VB>(st + L::V_OFF + ((kq * G + gg) * kWarp + lane) * VB,
                             src + gg * 8 * VB);
        }
    };

    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float bs[G][2];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) bs[gg][0] = bs[gg][1] = 0.f;
    const float sl2 = p.scale * 1.4426950408889634f;  // scores in base 2

#pragma unroll
    for (int i = 0; i < S - 1; ++i) {
        if (i < nmine) issue(i);
        cp_async_commit();
    }
    for (int i = 0; i < nmine; ++i) {
        if (i + S - 1 < nmine) issue(i + S - 1);
        cp_async_commit();
        cp_async_wait<S - 1>();  // tile i has landed
        const unsigned char *st = wsm + (i % S) * L::STAGE;
        const int ts = t0 + (warp + i * kAttWarps) * kAttTile;

        // scores: two accumulator chains over the k-steps
        float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < KC; ++c) {
            const uint4 k0 = *reinterpret_cast<const uint4 *>(
                st + L::K_OFF + (c * kWarp + lane) * 16);
            const uint4 k1 = *reinterpret_cast<const uint4 *>(
                st + L::K_OFF + ((KC + c) * kWarp + lane) * 16);
            mma_bf16(ca, k0.x, k1.x, k0.y, k1.y, qf[c].x, qf[c].y);
            mma_bf16(cb, k0.z, k1.z, k0.w, k1.w, qf[c].z, qf[c].w);
        }
        // x[kk][h]: key ts + 2g + kk against row 2t + h, masked to -inf
        float x[2][2];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int key = ts + 2 * g + kk;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                x[kk][h] = key < t1 && key < tm[h]
                               ? (ca[2 * kk + h] + cb[2 * kk + h]) * sl2
                               : -INFINITY;
        }
        float cr[2], pr[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float mt = fmaxf(x[0][h], x[1][h]);
#pragma unroll
            for (int off = 4; off < kWarp; off <<= 1)
                mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, off));
            const float mn = fmaxf(m[h], mt);
            cr[h] = mn == -INFINITY ? 1.f : ex2(m[h] - mn);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
                pr[kk][h] = x[kk][h] == -INFINITY ? 0.f : ex2(x[kk][h] - mn);
            l[h] = l[h] * cr[h] + pr[0][h] + pr[1][h];
            m[h] = mn;
        }
        if (!__all_sync(FULL, cr[0] == 1.f && cr[1] == 1.f)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                o[j][0] *= cr[0];
                o[j][1] *= cr[1];
                o[j][2] *= cr[0];
                o[j][3] *= cr[1];
            }
        }

        // scales and biases of keys 2g, 2g + 1, group gg
        float sc[2][G], bi[2][G];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const unsigned char *ss = st + L::S_OFF + (kk * kWarp + lane) * SB;
            const unsigned char *sb = st + L::B_OFF + (kk * kWarp + lane) * SB;
            if constexpr (G == 1) {
                const int64_t row = kv + min(ts + 2 * g + kk, t1 - 1);
                const int sh = (int)(row & 1) * 16;
                sc[kk][0] = bf16_bits_to_f32(
                    (uint16_t)(*reinterpret_cast<const uint32_t *>(ss) >> sh));
                bi[kk][0] = bf16_bits_to_f32(
                    (uint16_t)(*reinterpret_cast<const uint32_t *>(sb) >> sh));
            } else {
#pragma unroll
                for (int w = 0; w < G / 2; ++w) {
                    const uint32_t vs = reinterpret_cast<const uint32_t *>(ss)[w];
                    const uint32_t vb = reinterpret_cast<const uint32_t *>(sb)[w];
                    sc[kk][2 * w] = bf16_lo(vs);
                    sc[kk][2 * w + 1] = bf16_hi(vs);
                    bi[kk][2 * w] = bf16_lo(vb);
                    bi[kk][2 * w + 1] = bf16_hi(vb);
                }
            }
        }

#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
                bs[gg][h] = fmaf(pr[0][h], bi[0][gg],
                                 fmaf(pr[1][h], bi[1][gg], bs[gg][h] * cr[h]));
            // P' rows (keys 2g / 2g + 1) x columns (rows 2t, 2t + 1), then
            // transposed into the value product's B fragments
            const uint32_t pb0 = movmatrix_t(
                pack_bf16(pr[0][0] * sc[0][gg], pr[0][1] * sc[0][gg]));
            const uint32_t pb1 = movmatrix_t(
                pack_bf16(pr[1][0] * sc[1][gg], pr[1][1] * sc[1][gg]));
            const unsigned char *sv = st + L::V_OFF + (gg * kWarp + lane) * VB;
            constexpr int KQ = G * kWarp * VB;  // stride between the four keys
            if constexpr (BITS == 4) {
                // keys 4t, 4t+2 (k = 2t, 2t+1) and 4t+1, 4t+3 (k = 2t+8, 2t+9)
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(sv);
                const uint32_t wc = *reinterpret_cast<const uint32_t *>(sv + KQ);
                const uint32_t wb = *reinterpret_cast<const uint32_t *>(sv + 2 * KQ);
                const uint32_t wd = *reinterpret_cast<const uint32_t *>(sv + 3 * KQ);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    // byte jj of each word: dimensions 8g + 2jj (low nibble,
                    // m-row g) and 8g + 2jj + 1 (high nibble, m-row g + 8)
                    const uint32_t sel =
                        jj | (jj << 4) | ((4 + jj) << 8) | ((4 + jj) << 12);
                    const uint32_t rab = __byte_perm(wa, wb, sel);
                    const uint32_t rcd = __byte_perm(wc, wd, sel);
                    mma_bf16(o[4 * gg + jj], codes_bf16x2(rab), codes_bf16x2(rab >> 4),
                             codes_bf16x2(rcd), codes_bf16x2(rcd >> 4), pb0, pb1);
                }
            } else {
                // 8-bit codes as 16 * high nibble + low nibble: two products,
                // the high one against 16 P' (exact in bf16)
                const __nv_bfloat162 k16 = bits_bf2(0x41804180u);  // 16.0
                const uint32_t ph0 = bf2_bits(__hmul2(bits_bf2(pb0), k16));
                const uint32_t ph1 = bf2_bits(__hmul2(bits_bf2(pb1), k16));
                const uint2 wa = *reinterpret_cast<const uint2 *>(sv);
                const uint2 wc = *reinterpret_cast<const uint2 *>(sv + KQ);
                const uint2 wb = *reinterpret_cast<const uint2 *>(sv + 2 * KQ);
                const uint2 wd = *reinterpret_cast<const uint2 *>(sv + 3 * KQ);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    // bytes 2jj (m-row g) and 2jj + 1 (m-row g + 8)
                    const int e = 2 * (jj & 1);
                    const uint32_t sel =
                        e | ((e + 1) << 4) | ((4 + e) << 8) | ((5 + e) << 12);
                    const uint32_t rab =
                        __byte_perm(jj < 2 ? wa.x : wa.y, jj < 2 ? wb.x : wb.y, sel);
                    const uint32_t rcd =
                        __byte_perm(jj < 2 ? wc.x : wc.y, jj < 2 ? wd.x : wd.y, sel);
                    mma_bf16(o[4 * gg + jj], codes_bf16x2(rab), codes_bf16x2(rab >> 8),
                             codes_bf16x2(rcd), codes_bf16x2(rcd >> 8), pb0, pb1);
                    mma_bf16(o[4 * gg + jj], codes_bf16x2(rab >> 4),
                             codes_bf16x2(rab >> 12), codes_bf16x2(rcd >> 4),
                             codes_bf16x2(rcd >> 12), ph0, ph1);
                }
            }
        }
    }
    cp_async_wait<0>();

    // the lane's sums cover keys 2g, 2g + 1 of each tile: add over g
#pragma unroll
    for (int off = 4; off < kWarp; off <<= 1) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l[h] += __shfl_xor_sync(FULL, l[h], off);
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                bs[gg][h] += __shfl_xor_sync(FULL, bs[gg][h], off);
        }
    }
    // the warp's (unnormalized) output rows into its own ring: [row][D];
    // m-tile 4gg + jj holds dimensions 64gg + 8g + 2jj (+1 for m-row g + 8)
    __syncwarp();
    float *so = reinterpret_cast<float *>(wsm);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int d = 64 * (j / 4) + 8 * g + 2 * (j % 4);
        so[(2 * t) * D + d] = o[j][0];
        so[(2 * t + 1) * D + d] = o[j][1];
        so[(2 * t) * D + d + 1] = o[j][2];
        so[(2 * t + 1) * D + d + 1] = o[j][3];
    }
    if (g == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            s_m[warp][2 * t + h] = m[h];
            s_l[warp][2 * t + h] = l[h];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) s_b[warp][2 * t + h][gg] = bs[gg][h];
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kAttRows * (D + 2); e += blockDim.x) {
        const int i = e / (D + 2), c = e % (D + 2);
        if (i >= nlive) continue;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttWarps; ++w) mx = fmaxf(mx, s_m[w][i]);
        float val = 0.f;
        if (c == D) {
            val = mx;
        } else {
#pragma unroll
            for (int w = 0; w < kAttWarps; ++w) {
                const float f = s_m[w][i] == -INFINITY ? 0.f : ex2(s_m[w][i] - mx);
                const float *sow =
                    reinterpret_cast<const float *>(att_smem + w * L::WARP_BYTES);
                val += f * (c == D + 1 ? s_l[w][i] : sow[i * D + c] + s_b[w][i][c / 64]);
            }
        }
        const int r = rg * kAttRows + i;
        const int hq = hk * rep + r / p.Lq, lq = r % p.Lq;
        float *dst = p.part + ((((int64_t)b * p.Hq + hq) * p.Lq + lq) * p.nsplit +
                               split) * (D + 2);
        dst[c] = val;  // [0, D): output, D: max (base 2), D + 1: sum
    }
}

// out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits (the
// maxima are base-2 scores).  The splits' maxima and sums are read in
// parallel into shared memory first; each thread then adds its dimension
// over the splits with eight loads in flight.
template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(AttParams p) {
    __shared__ float s_f[kAttMaxSplits];  // 2^(m_s - M), 0 for empty splits
    __shared__ float s_red[D / kWarp];
    __shared__ float s_mx, s_den;
    if (threadIdx.x == 0) pdl_launch_dependents();
    pdl_wait_primary();  // the partials are the previous kernel's output
    const int64_t row = blockIdx.x;  // (b, hq, lq)
    const float *src = p.part + row * p.nsplit * (D + 2);
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x / kWarp;
    float mx = -INFINITY;
    for (int sp = threadIdx.x; sp < p.nsplit; sp += D) {
        const float ms = src[(int64_t)sp * (D + 2) + D];
        s_f[sp] = ms;
        mx = fmaxf(mx, ms);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = -INFINITY;
        for (int w = 0; w < D / kWarp; ++w) m = fmaxf(m, s_red[w]);
        s_mx = m;
    }
    __syncthreads();
    const float M = s_mx;
    float den = 0.f;
    for (int sp = threadIdx.x; sp < p.nsplit; sp += D) {
        const float ms = s_f[sp];
        const float f = ms == -INFINITY ? 0.f : ex2(ms - M);
        s_f[sp] = f;
        den += f * src[(int64_t)sp * (D + 2) + D + 1];
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    __syncthreads();  // s_red reuse, and every s_f written
    if (lane == 0) s_red[warp] = den;
    __syncthreads();
    if (threadIdx.x == 0) {
        float d = 0.f;
        for (int w = 0; w < D / kWarp; ++w) d += s_red[w];
        s_den = d;
    }
    __syncthreads();
    float num = 0.f;
    int sp = 0;
    for (; sp + 8 <= p.nsplit; sp += 8) {
        float ov[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) ov[u] = src[(int64_t)(sp + u) * (D + 2) + threadIdx.x];
#pragma unroll
        for (int u = 0; u < 8; ++u) num = fmaf(s_f[sp + u], ov[u], num);
    }
    for (; sp < p.nsplit; ++sp)
        num = fmaf(s_f[sp], src[(int64_t)sp * (D + 2) + threadIdx.x], num);
    p.out[row * D + threadIdx.x] = f32_to_bf16_bits(num / s_den);
}

// Splits per (batch, KV head, row group): one wave of blocks at the
// kernel's residency, at least one tile per warp in each split.
static int attn_splits(int64_t B, int Hkv, int rowgroups, int64_t T,
                       int blocks_per_sm) {
    const int64_t units = B * Hkv * rowgroups;
    int64_t s = ((int64_t)num_sms() * blocks_per_sm + units - 1) / units;
    const int64_t most = (T + kAttWarps * kAttTile - 1) / (kAttWarps * kAttTile);
    if (s > most) s = most;
    if (s < 1) s = 1;
    if (s > kAttMaxSplits) s = kAttMaxSplits;
    return (int)s;
}

static int attn_blocks_per_sm(int bits, int D) {
#define GWA_ATT(BB, DD) \
    if (bits == BB && D == DD) return AttLayout<BB, DD>::BLOCKS_PER_SM;
    GWA_ATT(4, 64) GWA_ATT(4, 128) GWA_ATT(4, 256)
    GWA_ATT(8, 64) GWA_ATT(8, 128) GWA_ATT(8, 256)
#undef GWA_ATT
    return 1;
}

// Opt a kernel in to more than 48 KB of dynamic shared memory (once per
// device).
static cudaError_t allow_smem(const void *kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<int, const void *>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(std::make_pair(dev, kernel))) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes);
    if (e != cudaSuccess) return e;
    done.insert(std::make_pair(dev, kernel));
    return cudaSuccess;
}

template <int BITS, int D>
static cudaError_t launch_attn_t(const AttParams &p, cudaStream_t st) {
    using L = AttLayout<BITS, D>;
    const void *kfn = reinterpret_cast<const void *>(attn_partial_kernel<BITS, D>);
    cudaError_t e = allow_smem(kfn, L::BYTES);
    if (e != cudaSuccess) return e;
    e = prefer_max_shared(kfn);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nsplit, (unsigned)(p.Hkv * p.rowgroups),
                       (unsigned)p.B);
    cfg.blockDim = dim3(kAttWarps * kWarp);
    cfg.dynamicSmemBytes = L::BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_partial_kernel<BITS, D>, p);
    if (e != cudaSuccess) return e;
    return launch_pdl(reinterpret_cast<const void *>(attn_combine_kernel<D>),
                      (unsigned)((int64_t)p.B * p.Hq * p.Lq), (unsigned)D, 0,
                      st, p);
}

cudaError_t launch_attention(const uint16_t *q, const uint16_t *k,
                             const uint32_t *vq, const uint16_t *vs,
                             const uint16_t *vb, uint16_t *out, float *part,
                             int B, int Hq, int Hkv, int Lq, int T, int D,
                             int bits, float scale, int causal,
                             cudaStream_t st) {
    AttParams p{};
    p.q = q; p.k = k; p.vq = vq; p.vs = vs; p.vb = vb; p.out = out;
    p.part = part;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Lq = Lq; p.T = T;
    p.rowgroups = (Hq / Hkv * Lq + kAttRows - 1) / kAttRows;
    p.nsplit = attn_splits(B, Hkv, p.rowgroups, T, attn_blocks_per_sm(bits, D));
    p.scale = scale;
    p.causal = causal;
#define GWA_ATT(BB, DD) \
    if (bits == BB && D == DD) return launch_attn_t<BB, DD>(p, st);
    GWA_ATT(4, 64) GWA_ATT(4, 128) GWA_ATT(4, 256)
    GWA_ATT(8, 64) GWA_ATT(8, 128) GWA_ATT(8, 256)
#undef GWA_ATT
    return cudaErrorInvalidValue;
}

// Workspace for the larger split count of the two code widths (the
// workspace query does not take the width).
size_t attention_workspace_bytes(int B, int Hq, int Hkv, int Lq, int T,
                                 int D) {
    const int rowgroups = (Hq / Hkv * Lq + kAttRows - 1) / kAttRows;
    const int ns = std::max(
        attn_splits(B, Hkv, rowgroups, T, attn_blocks_per_sm(4, D)),
        attn_splits(B, Hkv, rowgroups, T, attn_blocks_per_sm(8, D)));
    return (size_t)B * Hq * Lq * ns * (D + 2) * sizeof(float);
}

}  // namespace gwa
