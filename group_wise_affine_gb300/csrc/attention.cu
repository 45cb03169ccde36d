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
// Floats per (query row, split) partial: D outputs, the max and the sum,
// padded so each partial starts on 16 bytes.
template <int D>
constexpr int kAttPartStride = D + 4;

struct AttParams {
    const uint16_t *q;    // [B, Hq, Lq, D]
    const uint16_t *k;    // [B, Hkv, T, D]
    const uint32_t *vq;   // [B, Hkv, T, D*bits/32]
    const uint16_t *vs;   // [B, Hkv, T, D/64]
    const uint16_t *vb;
    uint16_t *out;        // [B, Hq, Lq, D]
    float *part;          // [B, Hq, Lq, nsplit, D + 4]
    int B, Hq, Hkv, Lq, T, nsplit, rowgroups;
    float scale;
    int causal;
};

// Resident blocks of kAttWarps warps with four ring stages of `stage` bytes
// in an SM's 228 KB (2 KB per block for the static buffers and the
// system's share), at most four.
constexpr int att_blocks(int stage) {
    return (228 * 1024) / (kAttWarps * 4 * stage + 2048) > 4
               ? 4
               : (228 * 1024) / (kAttWarps * 4 * stage + 2048);
}

// One warp's stage of the ring (one tile), in bytes.  Every item is laid
// out [item][lane] so a warp's copies and reads of one item are consecutive.
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
    static constexpr int S = 4;  // two tiles computed while two load
    static constexpr int BLOCKS_PER_SM = att_blocks(STAGE);
    static constexpr int WARP_BYTES = STAGE * S;
    static constexpr int BYTES = WARP_BYTES * kAttWarps;
    static_assert(kAttRows * D * 4 <= WARP_BYTES, "merge buffer fits the ring");
    static_assert(BLOCKS_PER_SM >= 1, "shared memory per SM");
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

// The 4-bit fields at bits 0-3 and 16-19 of x as a bf16 pair of 128 + q
// (0x4300 | q, exact); the 128 * sum of the weights it adds is taken back
// in the bias term.
__device__ __forceinline__ uint32_t codes_bf16x2(uint32_t x) {
    return (x & 0x000f000fu) | 0x43004300u;
}

// Bulk L2 prefetch of [ptr, ptr + bytes) by the copy engine (ptr and bytes
// multiples of 16).
__device__ __forceinline__ void prefetch_bulk_l2(const void *ptr, int bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes)
                 : "memory");
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
    __shared__ float s_f[kAttWarps][kAttRows];
    __shared__ float *s_dst[kAttRows];

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
    const int ntile = t1 > t0 ? (t1 - t0 + kAttTile - 1) / kAttTile : 0;
    const int nmine = ntile > warp ? (ntile - warp + kAttWarps - 1) / kAttWarps : 0;
    const int npair = (nmine + 1) / 2;  // an odd count ends on a masked tile
    if (threadIdx.x == 0) pdl_launch_dependents();
    // While the previous kernel finishes, pull the K and code rows of this
    // warp's first two tiles into L2.  A prefetch moves nothing into the
    // SM, so the copies made after the wait still see whatever that kernel
    // writes.  (The transfer into the SMs after the wait, not the DRAM
    // latency, dominates the first tiles, so this gains little when the
    // previous kernel is short.)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int ts = t0 + (warp + j * kAttWarps) * kAttTile;
        if (j < nmine) {
            const int nk = min(kAttTile, t1 - ts);
            const int64_t r0 = kv + ts;
            if (lane == 0) {  // K and code rows: 16-byte aligned, whole
                prefetch_bulk_l2(p.k + r0 * D, nk * D * 2);
                prefetch_bulk_l2(p.vq + r0 * WPR, nk * WPR * 4);
            }
        }
    }
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

    // Tile i of this warp: keys ts .. ts + 15.  The scores' row g is key
    // 2g and row g + 8 key 2g + 1 (the lane copies those two K rows and
    // their scales and biases); the value product's k = 2t, 2t + 1 are keys
    // 4t, 4t + 2 and k = 2t + 8, 2t + 9 keys 4t + 1, 4t + 3 (the lane copies
    // its 8 dimensions of each group of those four keys).  Keys past the
    // split are clamped to its last key and masked; a warp with an odd
    // number of tiles computes one more, wholly past the split, so that
    // tiles go in pairs.
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
    const int lim[2] = {min(t1, tm[0]), min(t1, tm[1])};
    // The running max m moves only when a score exceeds it by more than
    // 2^kLazy (weights up to 2^8: no overflow, no loss), so most tiles need
    // one vote instead of a max-reduction and a rescale.
    constexpr float kLazy = 8.f;
    // 128 * weight enters the value product with every code (once per
    // nibble product: 1 + 16 for 8-bit codes)
    constexpr float kCodeBias = BITS == 4 ? 128.f : 128.f * 17.f;

    if (npair > 0) {
        issue(0);
        issue(1);  // not part of the split when nmine == 1: masked
    }
    cp_async_commit();
    cp_async_commit();
    for (int it = 0; it < npair; ++it) {
        if (it + 1 < npair) {
            issue(2 * it + 2);
            issue(2 * it + 3);
        }
        cp_async_commit();
        cp_async_wait<1>();  // tiles 2it and 2it + 1 (one group) have landed
        const unsigned char *stg[2];
        stg[0] = wsm + ((2 * it) % S) * L::STAGE;
        stg[1] = stg[0] + L::STAGE;
        int ts[2];
        ts[0] = t0 + (warp + 2 * it * kAttWarps) * kAttTile;
        ts[1] = ts[0] + kAttWarps * kAttTile;

        // scores: two accumulator chains per tile over the k-steps
        float ca[2][4], cb[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) ca[u][e] = cb[u][e] = 0.f;
#pragma unroll
        for (int c = 0; c < KC; ++c) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint4 k0 = *reinterpret_cast<const uint4 *>(
                    stg[u] + L::K_OFF + (c * kWarp + lane) * 16);
                const uint4 k1 = *reinterpret_cast<const uint4 *>(
                    stg[u] + L::K_OFF + ((KC + c) * kWarp + lane) * 16);
                mma_bf16(ca[u], k0.x, k1.x, k0.y, k1.y, qf[c].x, qf[c].y);
                mma_bf16(cb[u], k0.z, k1.z, k0.w, k1.w, qf[c].z, qf[c].w);
            }
        }
        // x[u][kk][h]: key ts[u] + 2g + kk against row 2t + h, or -inf
        float x[2][2][2], lm[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int key = ts[u] + 2 * g + kk;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    x[u][kk][h] = key < lim[h]
                                      ? (ca[u][2 * kk + h] + cb[u][2 * kk + h]) * sl2
                                      : -INFINITY;
                    lm[h] = fmaxf(lm[h], x[u][kk][h]);
                }
            }
        if (__any_sync(FULL, lm[0] > m[0] + kLazy || lm[1] > m[1] + kLazy)) {
            float cr[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float mt = lm[h];
#pragma unroll
                for (int off = 4; off < kWarp; off <<= 1)
                    mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, off));
                const float mn = fmaxf(m[h], mt);
                cr[h] = mn == -INFINITY ? 1.f : ex2(m[h] - mn);
                m[h] = mn;
                l[h] *= cr[h];
#pragma unroll
                for (int gg = 0; gg < G; ++gg) bs[gg][h] *= cr[h];
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                o[j][0] *= cr[0];
                o[j][1] *= cr[1];
                o[j][2] *= cr[0];
                o[j][3] *= cr[1];
            }
        }
        float pr[2][2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    pr[u][kk][h] = x[u][kk][h] == -INFINITY ? 0.f : ex2(x[u][kk][h] - m[h]);
                    l[h] += pr[u][kk][h];
                }

        // scales and biases of keys 2g, 2g + 1 of each tile, group gg
        float sc[2][2][G], bi[2][2][G];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const unsigned char *ss = stg[u] + L::S_OFF + (kk * kWarp + lane) * SB;
                const unsigned char *sb = stg[u] + L::B_OFF + (kk * kWarp + lane) * SB;
                if constexpr (G == 1) {
                    const int64_t row = kv + min(ts[u] + 2 * g + kk, t1 - 1);
                    const int sh = (int)(row & 1) * 16;
                    sc[u][kk][0] = bf16_bits_to_f32(
                        (uint16_t)(*reinterpret_cast<const uint32_t *>(ss) >> sh));
                    bi[u][kk][0] = bf16_bits_to_f32(
                        (uint16_t)(*reinterpret_cast<const uint32_t *>(sb) >> sh));
                } else {
#pragma unroll
                    for (int w = 0; w < G / 2; ++w) {
                        const uint32_t vs = reinterpret_cast<const uint32_t *>(ss)[w];
                        const uint32_t vb = reinterpret_cast<const uint32_t *>(sb)[w];
                        sc[u][kk][2 * w] = bf16_lo(vs);
                        sc[u][kk][2 * w + 1] = bf16_hi(vs);
                        bi[u][kk][2 * w] = bf16_lo(vb);
                        bi[u][kk][2 * w + 1] = bf16_hi(vb);
                    }
                }
            }

#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            uint32_t pb[2][2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                // P' rows (keys 2g / 2g + 1) x columns (rows 2t, 2t + 1),
                // then transposed into the value product's B fragments
                const uint32_t x0 = pack_bf16(pr[u][0][0] * sc[u][0][gg],
                                              pr[u][0][1] * sc[u][0][gg]);
                const uint32_t x1 = pack_bf16(pr[u][1][0] * sc[u][1][gg],
                                              pr[u][1][1] * sc[u][1][gg]);
                // bias term, less the 128 * P' (as rounded) the codes carry
                bs[gg][0] = fmaf(pr[u][0][0], bi[u][0][gg],
                                 fmaf(pr[u][1][0], bi[u][1][gg],
                                      fmaf(-kCodeBias, bf16_lo(x0) + bf16_lo(x1),
                                           bs[gg][0])));
                bs[gg][1] = fmaf(pr[u][0][1], bi[u][0][gg],
                                 fmaf(pr[u][1][1], bi[u][1][gg],
                                      fmaf(-kCodeBias, bf16_hi(x0) + bf16_hi(x1),
                                           bs[gg][1])));
                pb[u][0] = movmatrix_t(x0);
                pb[u][1] = movmatrix_t(x1);
            }
            constexpr int KQ = G * kWarp * VB;  // stride between the four keys
            if constexpr (BITS == 4) {
                // keys 4t, 4t+2 (k = 2t, 2t+1) and 4t+1, 4t+3 (k = 2t+8, 2t+9)
                uint32_t wa[2], wb[2], wc[2], wd[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const unsigned char *sv = stg[u] + L::V_OFF + (gg * kWarp + lane) * VB;
                    wa[u] = *reinterpret_cast<const uint32_t *>(sv);
                    wc[u] = *reinterpret_cast<const uint32_t *>(sv + KQ);
                    wb[u] = *reinterpret_cast<const uint32_t *>(sv + 2 * KQ);
                    wd[u] = *reinterpret_cast<const uint32_t *>(sv + 3 * KQ);
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    // byte jj of each word: dimensions 8g + 2jj (low nibble,
                    // m-row g) and 8g + 2jj + 1 (high nibble, m-row g + 8)
                    const uint32_t sel =
                        jj | (jj << 4) | ((4 + jj) << 8) | ((4 + jj) << 12);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t rab = __byte_perm(wa[u], wb[u], sel);
                        const uint32_t rcd = __byte_perm(wc[u], wd[u], sel);
                        mma_bf16(o[4 * gg + jj], codes_bf16x2(rab), codes_bf16x2(rab >> 4),
                                 codes_bf16x2(rcd), codes_bf16x2(rcd >> 4), pb[u][0],
                                 pb[u][1]);
                    }
                }
            } else {
                // 8-bit codes as 16 * high nibble + low nibble: two products,
                // the high one against 16 P' (exact in bf16)
                const __nv_bfloat162 k16 = bits_bf2(0x41804180u);  // 16.0
                uint2 wa[2], wb[2], wc[2], wd[2];
                uint32_t ph[2][2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const unsigned char *sv = stg[u] + L::V_OFF + (gg * kWarp + lane) * VB;
                    wa[u] = *reinterpret_cast<const uint2 *>(sv);
                    wc[u] = *reinterpret_cast<const uint2 *>(sv + KQ);
                    wb[u] = *reinterpret_cast<const uint2 *>(sv + 2 * KQ);
                    wd[u] = *reinterpret_cast<const uint2 *>(sv + 3 * KQ);
                    ph[u][0] = bf2_bits(__hmul2(bits_bf2(pb[u][0]), k16));
                    ph[u][1] = bf2_bits(__hmul2(bits_bf2(pb[u][1]), k16));
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    // bytes 2jj (m-row g) and 2jj + 1 (m-row g + 8)
                    const int e = 2 * (jj & 1);
                    const uint32_t sel =
                        e | ((e + 1) << 4) | ((4 + e) << 8) | ((5 + e) << 12);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t rab = __byte_perm(jj < 2 ? wa[u].x : wa[u].y,
                                                         jj < 2 ? wb[u].x : wb[u].y, sel);
                        const uint32_t rcd = __byte_perm(jj < 2 ? wc[u].x : wc[u].y,
                                                         jj < 2 ? wd[u].x : wd[u].y, sel);
                        mma_bf16(o[4 * gg + jj], codes_bf16x2(rab), codes_bf16x2(rab >> 8),
                                 codes_bf16x2(rcd), codes_bf16x2(rcd >> 8), pb[u][0],
                                 pb[u][1]);
                        mma_bf16(o[4 * gg + jj], codes_bf16x2(rab >> 4),
                                 codes_bf16x2(rab >> 12), codes_bf16x2(rcd >> 4),
                                 codes_bf16x2(rcd >> 12), ph[u][0], ph[u][1]);
                    }
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
    // m-tile 4gg + jj holds dimensions 64gg + 8g + 2jj (and + 1, m-row g + 8)
    __syncwarp();
    float *so = reinterpret_cast<float *>(wsm);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int d = 64 * (j / 4) + 8 * g + 2 * (j % 4);
        *reinterpret_cast<float2 *>(so + (2 * t) * D + d) = make_float2(o[j][0], o[j][2]);
        *reinterpret_cast<float2 *>(so + (2 * t + 1) * D + d) =
            make_float2(o[j][1], o[j][3]);
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
    // per row: the warps' factors 2^(m_w - max) and the row's partial slot
    if (threadIdx.x < nlive) {
        const int i = threadIdx.x;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttWarps; ++w) mx = fmaxf(mx, s_m[w][i]);
        float den = 0.f;
#pragma unroll
        for (int w = 0; w < kAttWarps; ++w) {
            const float f = s_m[w][i] == -INFINITY ? 0.f : ex2(s_m[w][i] - mx);
            s_f[w][i] = f;
            den += f * s_l[w][i];
        }
        const int r = rg * kAttRows + i;
        const int hq = hk * rep + r / p.Lq, lq = r % p.Lq;
        float *dst = p.part + ((((int64_t)b * p.Hq + hq) * p.Lq + lq) * p.nsplit +
                               split) * kAttPartStride<D>;
        s_dst[i] = dst;
        dst[D] = mx;       // max (base 2)
        dst[D + 1] = den;  // sum
    }
    __syncthreads();
    constexpr int C4 = D / 4;  // float4 columns of a row
    for (int e = threadIdx.x; e < nlive * C4; e += blockDim.x) {
        const int i = e / C4, c4 = e % C4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kAttWarps; ++w) {
            const float f = s_f[w][i], bw = s_b[w][i][c4 / 16];
            const float4 v = reinterpret_cast<const float4 *>(
                att_smem + w * L::WARP_BYTES)[i * C4 + c4];
            acc.x = fmaf(f, v.x + bw, acc.x);
            acc.y = fmaf(f, v.y + bw, acc.y);
            acc.z = fmaf(f, v.z + bw, acc.z);
            acc.w = fmaf(f, v.w + bw, acc.w);
        }
        reinterpret_cast<float4 *>(s_dst[i])[c4] = acc;  // output [0, D)
    }
}

// out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits (the
// maxima are base-2 scores).  Every load of a row's partials is independent,
// so they are all issued up front: each thread's dimension for the first
// kCombineChunk splits into registers, and the splits' maxima and sums into
// shared memory, before the block reduces the maxima; further chunks (more
// than kCombineChunk splits) cost one more round trip each.
constexpr int kCombineChunk = 64;

template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(AttParams p) {
    __shared__ float s_f[kAttMaxSplits];  // m_s, then 2^(m_s - M) (0 if empty)
    __shared__ float s_ls[kAttMaxSplits];
    __shared__ float s_red[D / kWarp];
    __shared__ float s_mx, s_den;
    if (threadIdx.x == 0) pdl_launch_dependents();
    pdl_wait_primary();  // the partials are the previous kernel's output
    const int64_t row = blockIdx.x;  // (b, hq, lq)
    const int ns = p.nsplit;
    const float *src = p.part + row * ns * kAttPartStride<D>;
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x / kWarp;
    float ov[kCombineChunk];
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u)
        ov[u] = u < ns ? src[(int64_t)u * kAttPartStride<D> + threadIdx.x] : 0.f;
    float mx = -INFINITY;
    for (int sp = threadIdx.x; sp < ns; sp += D) {
        const float ms = src[(int64_t)sp * kAttPartStride<D> + D];
        s_ls[sp] = src[(int64_t)sp * kAttPartStride<D> + D + 1];
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
    for (int sp = threadIdx.x; sp < ns; sp += D) {
        const float ms = s_f[sp];
        const float f = ms == -INFINITY ? 0.f : ex2(ms - M);
        s_f[sp] = f;
        den += f * s_ls[sp];
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
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u)
        if (u < ns) num = fmaf(s_f[u], ov[u], num);
    for (int c0 = kCombineChunk; c0 < ns; c0 += kCombineChunk) {
#pragma unroll
        for (int u = 0; u < kCombineChunk; ++u)
            ov[u] = c0 + u < ns ? src[(int64_t)(c0 + u) * kAttPartStride<D> + threadIdx.x] : 0.f;
#pragma unroll
        for (int u = 0; u < kCombineChunk; ++u)
            if (c0 + u < ns) num = fmaf(s_f[c0 + u], ov[u], num);
    }
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
    const size_t stride = D == 64 ? kAttPartStride<64> : D == 128 ? kAttPartStride<128>
                                                        : kAttPartStride<256>;
    return (size_t)B * Hq * Lq * ns * stride * sizeof(float);
}

}  // namespace gwa
