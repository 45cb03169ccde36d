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
// from HBM once per KV head.  In a block each warp takes tiles of 32 keys:
// first a lane per key forms that key's scores with every query row (the
// scaled queries broadcast from shared memory), the rows' running max, sum
// and output are updated once per tile (fp32 online softmax), then the
// lanes split the head dimension (D/32 each) to dequantize each key's
// packed value row in registers and add it with the key's weight (taken by
// shuffle).  The warps merge in shared memory and the block writes (max,
// sum, output) per row and split to the workspace; a second kernel rescales
// and adds the splits and writes bf16.
#include "group_dot.cuh"
#include "internal.h"

namespace gwa {

constexpr int kAttRows = 8;     // query rows per block (power of two)
constexpr int kAttWarps = 4;

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

// The lane's DL codes of a packed value row (DL * BITS bits at bit
// lane * DL * BITS), widened into a 64-bit window.
template <int BITS, int DL>
__device__ __forceinline__ uint64_t lane_codes(const uint32_t *vrow, int lane) {
    constexpr int NB = DL * BITS / 8;  // bytes per lane: 1, 2, 4 or 8
    const unsigned char *b = reinterpret_cast<const unsigned char *>(vrow);
    if constexpr (NB == 1) return b[lane];
    else if constexpr (NB == 2) return reinterpret_cast<const uint16_t *>(b)[lane];
    else if constexpr (NB == 4) return reinterpret_cast<const uint32_t *>(b)[lane];
    else {
        const uint2 v = reinterpret_cast<const uint2 *>(b)[lane];
        return (uint64_t)v.x | ((uint64_t)v.y << 32);
    }
}

template <int BITS, int D>
__global__ void __launch_bounds__(kAttWarps * kWarp)
    attn_partial_kernel(AttParams p) {
    constexpr int DL = D / kWarp;  // dimensions per lane (value pass)
    constexpr int WPR = D * BITS / 32;
    constexpr uint64_t MASK = (1ull << BITS) - 1ull;
    __shared__ __align__(16) float s_q[kAttRows][D];  // scaled queries
    __shared__ float s_m[kAttWarps][kAttRows], s_l[kAttWarps][kAttRows];
    __shared__ float s_o[kAttWarps][kAttRows][D];

    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x / kWarp;
    const int split = blockIdx.x;
    const int hk = blockIdx.y / p.rowgroups, rg = blockIdx.y % p.rowgroups;
    const int b = blockIdx.z;
    const int rep = p.Hq / p.Hkv;
    const int nrows = rep * p.Lq;  // query rows of this KV head
    const int nlive = min(kAttRows, nrows - rg * kAttRows);
    const int64_t t0 = (int64_t)p.T * split / p.nsplit;
    const int64_t t1 = (int64_t)p.T * (split + 1) / p.nsplit;
    if (threadIdx.x == 0) pdl_launch_dependents();
    pdl_wait_primary();  // q, k, v may come from the previous kernel

    int tmax[kAttRows];  // keys [0, tmax) visible to row i
#pragma unroll
    for (int i = 0; i < kAttRows; ++i) {
        const int r = rg * kAttRows + i;
        const int lq = i < nlive ? r % p.Lq : 0;
        tmax[i] = i >= nlive ? 0 : p.causal ? p.T - p.Lq + lq + 1 : p.T;
    }
    for (int e = threadIdx.x; e < kAttRows * D; e += blockDim.x) {
        const int i = e / D, d = e % D;
        float v = 0.f;
        if (i < nlive) {
            const int r = rg * kAttRows + i;
            const int hq = hk * rep + r / p.Lq, lq = r % p.Lq;
            v = bf16_bits_to_f32(
                    p.q[(((int64_t)b * p.Hq + hq) * p.Lq + lq) * D + d]) * p.scale;
        }
        s_q[i][d] = v;
    }
    __syncthreads();

    float m[kAttRows], l[kAttRows], o[kAttRows][DL];
#pragma unroll
    for (int i = 0; i < kAttRows; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int j = 0; j < DL; ++j) o[i][j] = 0.f;
    }
    const int64_t kv = ((int64_t)b * p.Hkv + hk) * p.T;  // first key row
    const int g = lane * DL / 64;                        // value pass group
    // a warp takes tiles of 32 keys: lane = key for the scores, then lane =
    // dimensions for the values
    for (int64_t tt = t0 + (int64_t)warp * kWarp; tt < t1;
         tt += (int64_t)kAttWarps * kWarp) {
        const int64_t key = tt + lane;
        const bool kin = key < t1;
        float sc[kAttRows];
#pragma unroll
        for (int i = 0; i < kAttRows; ++i) sc[i] = 0.f;
        if (kin) {
            const uint4 *kr = reinterpret_cast<const uint4 *>(p.k + (kv + key) * D);
#pragma unroll 4
            for (int c = 0; c < D / 8; ++c) {
                const uint4 u = kr[c];
                const float kf[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y),
                                     bf16_hi(u.y), bf16_lo(u.z), bf16_hi(u.z),
                                     bf16_lo(u.w), bf16_hi(u.w)};
#pragma unroll
                for (int i = 0; i < kAttRows; ++i) {
                    if (i >= nlive) break;
                    const float4 qa = *reinterpret_cast<const float4 *>(&s_q[i][8 * c]);
                    const float4 qb = *reinterpret_cast<const float4 *>(&s_q[i][8 * c + 4]);
                    float a = sc[i];
                    a = fmaf(qa.x, kf[0], a); a = fmaf(qa.y, kf[1], a);
                    a = fmaf(qa.z, kf[2], a); a = fmaf(qa.w, kf[3], a);
                    a = fmaf(qb.x, kf[4], a); a = fmaf(qb.y, kf[5], a);
                    a = fmaf(qb.z, kf[6], a); a = fmaf(qb.w, kf[7], a);
                    sc[i] = a;
                }
            }
        }
        // per row: the tile's max and sum, the running state rescaled once
        float pr[kAttRows];
#pragma unroll
        for (int i = 0; i < kAttRows; ++i) {
            pr[i] = 0.f;
            if (i >= nlive) continue;  // uniform
            const float s = kin && key < tmax[i] ? sc[i] : -INFINITY;
            float mt = s;
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1)
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o2));
            if (mt == -INFINITY) continue;  // no visible key in the tile
            const float mn = fmaxf(m[i], mt);
            const float pw = s == -INFINITY ? 0.f : __expf(s - mn);
            float ps = pw;
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1)
                ps += __shfl_xor_sync(0xffffffffu, ps, o2);
            const float corr = __expf(m[i] - mn);  // 0 while m = -inf
            l[i] = l[i] * corr + ps;
#pragma unroll
            for (int j = 0; j < DL; ++j) o[i][j] *= corr;
            m[i] = mn;
            pr[i] = pw;
        }
        // values: each key of the tile, dequantized by the lanes' dimensions
        const int nk = (int)min((int64_t)kWarp, t1 - tt);
        for (int j = 0; j < nk; ++j) {
            const int64_t row = kv + tt + j;
            const uint64_t codes = lane_codes<BITS, DL>(p.vq + row * WPR, lane);
            const float vsc = bf16_bits_to_f32(p.vs[row * (D / 64) + g]);
            const float vbi = bf16_bits_to_f32(p.vb[row * (D / 64) + g]);
            float v[DL];
#pragma unroll
            for (int d = 0; d < DL; ++d)
                v[d] = fmaf(vsc, (float)((codes >> (BITS * d)) & MASK), vbi);
#pragma unroll
            for (int i = 0; i < kAttRows; ++i) {
                if (i >= nlive) break;
                const float pj = __shfl_sync(0xffffffffu, pr[i], j);
#pragma unroll
                for (int d = 0; d < DL; ++d) o[i][d] = fmaf(pj, v[d], o[i][d]);
            }
        }
    }

    // merge the warps: each writes its state, then the block combines
#pragma unroll
    for (int i = 0; i < kAttRows; ++i) {
        if (lane == 0) {
            s_m[warp][i] = m[i];
            s_l[warp][i] = l[i];
        }
#pragma unroll
        for (int j = 0; j < DL; ++j) s_o[warp][i][lane * DL + j] = o[i][j];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kAttRows * (D + 2); e += blockDim.x) {
        const int i = e / (D + 2), c = e % (D + 2);
        if (i >= nlive) continue;
        const int r = rg * kAttRows + i;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttWarps; ++w) mx = fmaxf(mx, s_m[w][i]);
        float val = 0.f;
        if (c == D) {
            val = mx;
        } else {
#pragma unroll
            for (int w = 0; w < kAttWarps; ++w) {
                const float f = s_m[w][i] == -INFINITY ? 0.f : __expf(s_m[w][i] - mx);
                val += f * (c == D + 1 ? s_l[w][i] : s_o[w][i][c]);
            }
        }
        const int hq = hk * rep + r / p.Lq, lq = r % p.Lq;
        float *dst = p.part + ((((int64_t)b * p.Hq + hq) * p.Lq + lq) * p.nsplit +
                               split) * (D + 2);
        dst[c] = val;  // [0, D): output, D: max, D + 1: sum
    }
}

// out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s over the splits.  The
// splits' maxima and sums are read in parallel into shared memory first;
// each thread then adds its dimension over the splits with eight loads in
// flight.
constexpr int kAttMaxSplits = 1024;

template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(AttParams p) {
    __shared__ float s_f[kAttMaxSplits];  // e^(m_s - M), 0 for empty splits
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
        const float f = ms == -INFINITY ? 0.f : __expf(ms - M);
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

int attn_splits(int64_t B, int Hkv, int rowgroups, int64_t T) {
    // about four blocks per SM, at least a tile of 32 keys per warp a split
    int64_t s = ((int64_t)num_sms() * 4 + B * Hkv * rowgroups - 1) /
                (B * Hkv * rowgroups);
    const int64_t most = (T + kAttWarps * kWarp - 1) / (kAttWarps * kWarp);
    if (s > most) s = most;
    if (s < 1) s = 1;
    if (s > kAttMaxSplits) s = kAttMaxSplits;
    return (int)s;
}

template <int BITS, int D>
static cudaError_t launch_attn_t(const AttParams &p, cudaStream_t st) {
    const dim3 grid((unsigned)p.nsplit, (unsigned)(p.Hkv * p.rowgroups),
                    (unsigned)p.B);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kAttWarps * kWarp);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, attn_partial_kernel<BITS, D>, p);
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
    p.nsplit = attn_splits(B, Hkv, p.rowgroups, T);
    p.scale = scale;
    p.causal = causal;
#define GWA_ATT(BB, DD) \
    if (bits == BB && D == DD) return launch_attn_t<BB, DD>(p, st);
    GWA_ATT(4, 64) GWA_ATT(4, 128) GWA_ATT(4, 256)
    GWA_ATT(8, 64) GWA_ATT(8, 128) GWA_ATT(8, 256)
#undef GWA_ATT
    return cudaErrorInvalidValue;
}

size_t attention_workspace_bytes(int B, int Hq, int Hkv, int Lq, int T,
                                 int D) {
    const int rowgroups = (Hq / Hkv * Lq + kAttRows - 1) / kAttRows;
    const int ns = attn_splits(B, Hkv, rowgroups, T);
    return (size_t)B * Hq * Lq * ns * (D + 2) * sizeof(float);
}

}  // namespace gwa
