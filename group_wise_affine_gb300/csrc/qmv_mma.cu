// Decode kernel for 5..8 tokens on the tensor cores (u4/u8 codes, groups of
// 64; rows of 512..5120 inputs on one CTA, longer rows of a plain projection
// cut along K over a thread-block cluster): the same weight stream as the streaming
// decode kernel (a producer thread copies the rows of a CTA's units into a
// shared-memory ring with the bulk-copy engine), but the consumers form the
// products with warp-level bf16 MMAs (m16n8k16, fp32 accumulation):
//
//   C = X W^T     m = the tokens (8 of the 16 used), n = 8 weight rows,
//                 k = 16 inputs,
//
// per group of 64 inputs, then y += scale * (C - 128 X_g) + bias * X_g in
// fp32, X_g the group's activation sum.  Codes enter as the exact bf16
// 128 + q (0x4300 | q); u8 codes as their two nibbles in two products (the
// high one counted 16 times), each made exact by subtracting 128 in bf16.
// Activations are exact in bf16, so every product is exact and only the
// accumulation rounds.
//
// Work layout: a stage holds 8 units (rows, or gate/up or rotary pairs) of
// whole rows.  Consumer warp w owns inputs [512 w, 512 w + 512) of every
// row: eight groups, whose activation fragments (the 16 of each group its
// lane's k slice needs, for the lane's token) it keeps in registers for the
// whole kernel.  Per stage and group it reads its lane's 8 (u4) or 16 (u8)
// code bytes of weight row g, forms the B fragments, runs four (eight) MMAs
// into a fresh accumulator and folds it into the per-row totals with the
// row's scale and bias; the warps' totals go to per-warp slots that the
// epilogue adds in a fixed order (plain, sections with bias, SiLU(gate)*up,
// or the rotary embedding from p.rope_cs).
//
// Measured on the 27648 x 5120 gate+up weight: 36.9 us for 8 tokens in one
// pass (the streaming kernel streams the weights twice: ~72 us), but only
// level with the streaming kernel at 4 tokens (35.1 against 36.3 us), so it
// serves 5..8 tokens.  (Those figures predate the padded row stride below,
// which removed the eight-way bank conflicts of the B-fragment reads: QKV
// at 8 tokens 11.8 -> 10.9 us, gate+up unchanged.)
//
// k order: within a group, lane t's k-slice of k-step s (logical k 2t, 2t+1,
// 2t+8, 2t+9) is the nibbles (j, j+4) and (j+1, j+5), j = 2 (s & 1), of word
// 2t + s/2 (u4), or the low/high nibbles of bytes (0, 2) and (1, 3) of word
// 4t + s (u8), so both operands come from 16 contiguous inputs per lane.
// Formulas and sources as in qmv.cu ("Sanctum-MLX"; "The Cathedral Doubled
// Itself", "The two fusions"; "saragossa", "Quantization formats").
#include <cuda_bf16.h>


#include "cluster.cuh"
#include "common.cuh"
#include "internal.h"

namespace gwa {

static __device__ unsigned int g_mma_timeouts;

constexpr int kMmaUnits = 8;          // units per stage: the MMAs' n
// Padding after each row in a stage.  The eight rows of an MMA are read at
// the same offset, four lanes a row (u4 8 bytes, u8 16 bytes each); rows a
// multiple of 128 bytes apart would put all eight in the same banks, so a
// row's stride is its bytes plus 32 (u4) or 64 (u8): the reads then take
// the two (four) wavefronts their 256 (512) bytes need.
template <int BITS>
constexpr uint32_t kMmaRowPad = BITS == 4 ? 32u : 64u;
constexpr int kMmaGroupsPerWarp = 8;  // 512 inputs per consumer warp
constexpr int kMmaMaxWarps = 10;      // K <= 5120
constexpr int kMmaTokens = 8;
constexpr size_t kMmaRingTarget = 160 * 1024;

enum MmaMode { kMPlain = 0, kMSections = 1, kMGateUp = 2, kMRope = 3 };

// d += a b, bf16 m16n8k16 with the A rows 8..15 zero.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// The 4-bit fields at bits 0-3 and 16-19 of v as the bf16 pair 128 + q.
__device__ __forceinline__ uint32_t nib_pair(uint32_t v) {
    return (v & 0x000f000fu) | 0x43004300u;
}
// The same minus 128: the exact bf16 pair q.
__device__ __forceinline__ uint32_t nib_pair_exact(uint32_t v) {
    const uint32_t a = nib_pair(v);
    const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                     __floats2bfloat162_rn(128.f, 128.f));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Per-lane activation state: the A fragments (a0, a2) of the lane's token
// for every k-step of the warp's eight groups, and the groups' sums.
struct MmaX {
    uint32_t a[kMmaGroupsPerWarp][4][2];
    float xs[kMmaGroupsPerWarp];
};

// Loads the 16 inputs [16 t, 16 t + 16) of each of the warp's groups for
// token g (zeros for g >= M) and arranges them in the k order above.
template <int BITS>
__device__ __forceinline__ void mma_load_x(const uint16_t *__restrict__ x, int M,
                                           int K, int warp, int g, int t,
                                           MmaX &xr) {
#pragma unroll
    for (int gi = 0; gi < kMmaGroupsPerWarp; ++gi) {
        uint32_t w[8];
        if (g < M) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                x + (int64_t)g * K + (int64_t)(warp * kMmaGroupsPerWarp + gi) * kGroup +
                16 * t);
            const uint4 u0 = src[0], u1 = src[1];
            w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
            w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0u;
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += bf16_lo(w[i]) + bf16_hi(w[i]);
        // the group's sum: the four lanes t of token g
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        xr.xs[gi] = s;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t lo, hi;  // local indices of the pairs (l, l + d)
            if constexpr (BITS == 4) {
                // inputs 8 (ks/2) + j + {0, 4} and + {1, 5}, j = 2 (ks & 1)
                const int l = 8 * (ks >> 1) + 2 * (ks & 1);
                lo = __byte_perm(w[l / 2], w[l / 2 + 2], 0x5410);
                hi = __byte_perm(w[l / 2], w[l / 2 + 2], 0x7632);
            } else {
                // inputs 4 ks + {0, 2} and + {1, 3}
                lo = __byte_perm(w[2 * ks], w[2 * ks + 1], 0x5410);
                hi = __byte_perm(w[2 * ks], w[2 * ks + 1], 0x7632);
            }
            xr.a[gi][ks][0] = lo;
            xr.a[gi][ks][1] = hi;
        }
        // one group's loads at a time (registers)
        asm volatile("" ::: "memory");
    }
}

// 168 registers: up to 11 warps (10 consumers and the producer) per CTA.
// KS > 1: rows longer than 5120 inputs, cut along K over a cluster of KS
// CTAs.  Rank r streams inputs [r K/KS, (r+1) K/KS) of the cluster's rows
// (one bulk copy per row segment) and keeps those activations; the ranks'
// partial sums meet in rank 0 over distributed shared memory, added in rank
// order, and rank 0 runs the epilogue.
template <int BITS, int MODE, int KS>
__global__ void __maxnreg__(168)
    qmv_mma_kernel(DenseParams p, int stages, int64_t units, int nw) {
    constexpr int HALVES = (MODE == kMGateUp || MODE == kMRope) ? 2 : 1;
    constexpr int GB = BITS * 8;  // code bytes per row and group
    constexpr int ups = kMmaUnits;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int ncons = nw * kWarp;
    const int lane = tid & (kWarp - 1), warp = tid / kWarp;
    const int M = p.M;
    const int rank = KS > 1 ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / KS, ncl = gridDim.x / KS;
    const int Ks = p.K / KS;      // inputs of a row this CTA covers
    const int Gs = Ks / kGroup;   // their groups
    // a row's share in a stage; whole rows in memory
    const uint32_t rowbytes = (uint32_t)Ks * BITS / 8;
    const uint32_t sbrow = (uint32_t)Gs * 2;
    const uint32_t growbytes = (uint32_t)p.K * BITS / 8;
    const uint32_t gsbrow = (uint32_t)p.G * 2;
    const uint32_t rows_stage = (uint32_t)(HALVES * ups);
    const uint32_t rowstride = rowbytes + kMmaRowPad<BITS>;
    const uint32_t stage_bytes = rows_stage * (rowstride + 2 * sbrow);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    uint64_t *empty = full + stages;
    float *red = reinterpret_cast<float *>(empty + stages);
    __shared__ int s_issued, s_consumed;

    // rope: whole stages per CTA (8 divides d/2), so no stage crosses a head
    const int64_t ualign = MODE == kMRope ? ups : 1;
    const int64_t u0 = units / ualign * cid / ncl * ualign;
    const int64_t u1 = units / ualign * (cid + 1) / ncl * ualign;
    const int nu = (int)(u1 - u0);
    const int nst = (nu + ups - 1) / ups;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nw);
        }
        fence_mbar_init();
        s_issued = 0;
        s_consumed = nst;
        pdl_launch_dependents();
    }
    __syncthreads();

    if (tid >= ncons) {
        // ------------------------------------------------ producer
        if (tid == ncons) {
            const unsigned char *wq = reinterpret_cast<const unsigned char *>(p.wq);
            const unsigned char *sc = reinterpret_cast<const unsigned char *>(p.sc);
            const unsigned char *bi = reinterpret_cast<const unsigned char *>(p.bi);
            for (int st = 0; st < nst; ++st) {
                const int s = st % stages;
                // weights are never written by this library's kernels: the
                // first `stages` stages are fetched before the wait
                if (st == stages) pdl_wait_primary();
                if (st >= stages && !mbar_wait(&empty[s], ((st / stages) & 1) ^ 1)) {
                    atomicAdd(&g_mma_timeouts, 1u);
                    break;
                }
                const int64_t ua = u0 + (int64_t)st * ups;
                const int n = (int)min((int64_t)ups, u1 - ua);
                unsigned char *base = smem + (size_t)s * stage_bytes;
                unsigned char *dsc = base + rows_stage * rowstride;
                unsigned char *dbi = dsc + rows_stage * sbrow;
                mbar_expect_tx(&full[s], (uint32_t)(HALVES * n) * (rowbytes + 2 * sbrow));
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    const int64_t r = MODE == kMRope ? rope_pair_row(ua, h, p.rope_hd)
                                                     : ua + (h ? p.I : 0);
                    if constexpr (KS == 1) {
                        // a copy per row (padded strides), one for the
                        // stage's scales and one for its biases
                        for (int i = 0; i < n; ++i)
                            bulk_g2s(base + (uint32_t)(h * ups + i) * rowstride,
                                     wq + (r + i) * rowbytes, rowbytes, &full[s]);
                        bulk_g2s(dsc + h * ups * sbrow, sc + r * sbrow, n * sbrow,
                                 &full[s]);
                        bulk_g2s(dbi + h * ups * sbrow, bi + r * sbrow, n * sbrow,
                                 &full[s]);
                    } else {
                        // this rank's segment of each row
                        for (int i = 0; i < n; ++i) {
                            const int64_t ri = r + i;
                            const uint32_t d = (uint32_t)(h * ups + i);
                            bulk_g2s(base + d * rowstride,
                                     wq + ri * growbytes + (uint32_t)rank * rowbytes,
                                     rowbytes, &full[s]);
                            bulk_g2s(dsc + d * sbrow,
                                     sc + ri * gsbrow + (uint32_t)rank * sbrow, sbrow,
                                     &full[s]);
                            bulk_g2s(dbi + d * sbrow,
                                     bi + ri * gsbrow + (uint32_t)rank * sbrow, sbrow,
                                     &full[s]);
                        }
                    }
                }
                s_issued = st + 1;
            }
        }
    } else {
        // ------------------------------------------------ consumers
        const int g = lane >> 2, t = lane & 3;  // token / weight row, k slice
        const int gbase = warp * kMmaGroupsPerWarp;
        MmaX xr;
        pdl_wait_primary();  // x may be the previous kernel's output
        mma_load_x<BITS>(p.x + (int64_t)rank * Ks, M, p.K, warp, g, t, xr);
        for (int st = 0; st < nst; ++st) {
            const int s = st % stages;
            if (!mbar_wait(&full[s], (st / stages) & 1)) {
                atomicAdd(&g_mma_timeouts, 1u);
                atomicMin(&s_consumed, st);
                break;
            }
            const int64_t ua = u0 + (int64_t)st * ups;
            const int n = (int)min((int64_t)ups, u1 - ua);
            const unsigned char *base = smem + (uint32_t)s * stage_bytes;
            const unsigned char *scb = base + rows_stage * rowstride;
            const unsigned char *bib = scb + rows_stage * sbrow;
            // rows past the stage's end hold stale data: their columns of
            // the products are dropped below
            float acc[HALVES][2];
#pragma unroll
            for (int h = 0; h < HALVES; ++h) acc[h][0] = acc[h][1] = 0.f;
#pragma unroll
            for (int gi = 0; gi < kMmaGroupsPerWarp; ++gi) {
                const int gg = gbase + gi;
                const float xs = xr.xs[gi];
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    // lane (g, t) supplies weight row g's k slice t ...
                    const unsigned char *wr = base + (uint32_t)(h * ups + g) * rowstride +
                                              (uint32_t)gg * GB + (uint32_t)t * (GB / 4);
                    float c[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (BITS == 4) {
                        const uint2 wv = *reinterpret_cast<const uint2 *>(wr);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint32_t word = ks < 2 ? wv.x : wv.y;
                            const int j = 2 * (ks & 1);
                            mma16816(c, xr.a[gi][ks][0], xr.a[gi][ks][1],
                                     nib_pair(word >> (4 * j)), nib_pair(word >> (4 * j + 4)));
                        }
                    } else {
                        const uint4 wv = *reinterpret_cast<const uint4 *>(wr);
                        float ch[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint32_t word = ks == 0   ? wv.x
                                                  : ks == 1 ? wv.y
                                                  : ks == 2 ? wv.z
                                                            : wv.w;
                            mma16816(c, xr.a[gi][ks][0], xr.a[gi][ks][1],
                                     nib_pair_exact(word), nib_pair_exact(word >> 8));
                            mma16816(ch, xr.a[gi][ks][0], xr.a[gi][ks][1],
                                     nib_pair_exact(word >> 4), nib_pair_exact(word >> 12));
                        }
                        c[0] = fmaf(16.f, ch[0], c[0]);
                        c[1] = fmaf(16.f, ch[1], c[1]);
                    }
                    // ... and gets the products of token g with rows 2t, 2t + 1
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        const uint32_t so = ((uint32_t)(h * ups + 2 * t + v) * Gs + gg) * 2u;
                        const float sv =
                            bf16_bits_to_f32(*reinterpret_cast<const uint16_t *>(scb + so));
                        const float bv =
                            bf16_bits_to_f32(*reinterpret_cast<const uint16_t *>(bib + so));
                        const float cv = BITS == 4 ? fmaf(-128.f, xs, c[v]) : c[v];
                        acc[h][v] = fmaf(sv, cv, fmaf(bv, xs, acc[h][v]));
                    }
                    // keep the next half's and group's loads after this
                    // one (registers)
                    asm volatile("" ::: "memory");
                }
            }
            // every lane's reads of this stage are done: release the slot
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (g < M) {
#pragma unroll
                for (int h = 0; h < HALVES; ++h)
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        const int u = 2 * t + v;
                        if (u < n)
                            red[(((st * ups + u) * HALVES + h) * M + g) * nw + warp] =
                                acc[h][v];
                    }
            }
        }
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
    if constexpr (KS > 1) {
        // this CTA's sum over its warps, in place of the first warp's slot
        for (int i = tid; i < nu * HALVES * M; i += blockDim.x) {
            float v = 0.f;
            for (int w = 0; w < nw; ++w) v += red[i * nw + w];
            red[i * nw] = v;
        }
        cluster_sync_all();
    }
    // the warps' slots of an output (the ranks' sums), added in a fixed order
    auto total = [&](int idx) {
        float v = 0.f;
        if constexpr (KS > 1) {
            float part[KS];  // all ranks' loads in flight at once
#pragma unroll
            for (int q = 0; q < KS; ++q)
                part[q] = ld_cluster_f32(red + idx * nw, (uint32_t)q);
#pragma unroll
            for (int q = 0; q < KS; ++q) v += part[q];
        } else {
            for (int w = 0; w < nw; ++w) v += red[idx * nw + w];
        }
        return v;
    };
    for (int i = tid; i < (rank == 0 ? nu * M : 0); i += blockDim.x) {
        const int lu = i / M, m = i % M;
        const int64_t n = u0 + lu;
        if constexpr (MODE == kMGateUp) {
            const float gv = total((lu * 2 + 0) * M + m);
            const float uv = total((lu * 2 + 1) * M + m);
            p.y[(int64_t)m * p.I + n] = f32_to_bf16_bits(gv / (1.0f + __expf(-gv)) * uv);
        } else if constexpr (MODE == kMRope) {
            const int half = p.rope_hd / 2;
            float a = total((lu * 2 + 0) * M + m);
            float b = total((lu * 2 + 1) * M + m);
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
                const float2 cs = p.rope_cs[(int64_t)m * half + (int)(n % half)];
                const float a2 = a * cs.x - b * cs.y;
                b = b * cs.x + a * cs.y;
                a = a2;
            }
            uint16_t *o = p.sec_out[s] + (int64_t)m * size + j;
            o[0] = f32_to_bf16_bits(a);
            o[half] = f32_to_bf16_bits(b);
        } else if constexpr (MODE == kMPlain) {
            p.y[(int64_t)m * p.N + n] = f32_to_bf16_bits(total(lu * M + m));
        } else {
            int s = 0;
            while (s + 1 < p.nsec && n >= p.sec_start[s + 1]) ++s;
            const int64_t j = n - p.sec_start[s];
            const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
            float val = total(lu * M + m);
            if (p.sec_bias[s]) val += bf16_bits_to_f32(p.sec_bias[s][j]);
            p.sec_out[s][(int64_t)m * size + j] = f32_to_bf16_bits(val);
        }
    }
    // no CTA leaves while rank 0 still reads its sums
    if constexpr (KS > 1) cluster_sync_all();
}

// ------------------------------------------------------------ host side

template <int BITS, int MODE, int KS>
static cudaError_t launch_mma_t(const DenseParams &p, cudaStream_t st, bool *used) {
    constexpr int HALVES = (MODE == kMGateUp || MODE == kMRope) ? 2 : 1;
    const int64_t units = MODE == kMGateUp ? p.I : MODE == kMRope ? p.N / 2 : p.N;
    if (units <= 0) return cudaSuccess;
    if (MODE == kMRope && (p.rope_hd / 2) % kMmaUnits != 0)
        return cudaSuccess;  // not used: stages would cross heads
    const int Ks = p.K / KS;
    const int nw = Ks / (kGroup * kMmaGroupsPerWarp);
    const int threads = (nw + 1) * kWarp;
    const size_t rowbytes = (size_t)Ks * BITS / 8;
    const size_t sbrow = (size_t)(Ks / kGroup) * 2;
    const size_t stage_bytes =
        (size_t)HALVES * kMmaUnits * (rowbytes + kMmaRowPad<BITS> + 2 * sbrow);
    const int64_t ualign = MODE == kMRope ? kMmaUnits : 1;
    int ncl = num_sms() / KS;  // clusters (CTAs when KS = 1)
    if ((int64_t)ncl > units / ualign) ncl = (int)(units / ualign);
    if (ncl < 1) return cudaSuccess;
    int stages = 0;
    size_t smem = 0;
    // ring stages and shared memory for ncl clusters (false: does not fit)
    auto plan = [&](int n) {
        const int64_t umax = (units / ualign + n - 1) / n * ualign;
        const size_t red_bytes = (size_t)umax * HALVES * p.M * nw * 4;
        if (red_bytes + 2 * (stage_bytes + 16) > kMaxDynSmem) return false;
        stages = (int)((kMaxDynSmem - red_bytes) / (stage_bytes + 16));
        const int cap = (int)(kMmaRingTarget / stage_bytes);
        if (stages > cap) stages = cap;
        if (stages > 8) stages = 8;
        if (stages < 2) stages = 2;
        smem = stages * (stage_bytes + 16) + red_bytes;
        return true;
    };
    if (!plan(ncl)) return cudaSuccess;
    auto kern = qmv_mma_kernel<BITS, MODE, KS>;
    int dummy = 0;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern), threads, smem,
                                   &dummy);
    if (e != cudaSuccess) return e;
    if constexpr (KS > 1) {
        // one wave: no more clusters than the GPU keeps resident
        const int res = resident_clusters(reinterpret_cast<const void *>(kern), KS,
                                              threads, smem);
        if (res < 1) return cudaSuccess;
        if (res < ncl) {
            ncl = res;
            if (!plan(ncl)) return cudaSuccess;
            e = occupancy_grid(reinterpret_cast<const void *>(kern), threads, smem,
                               &dummy);
            if (e != cudaSuccess) return e;
        }
        *used = true;
        return launch_pdl_cluster(reinterpret_cast<const void *>(kern),
                                  (unsigned)(ncl * KS), (unsigned)KS, (unsigned)threads,
                                  smem, st, p, stages, units, nw);
    }
    *used = true;
    return launch_pdl(reinterpret_cast<const void *>(kern), (unsigned)ncl,
                      (unsigned)threads, smem, st, p, stages, units, nw);
}

static bool mma_aligned16(const void *q) {
    return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
}

constexpr int kMmaMaxSplit = 4;  // CTAs per cluster along K

// Runs the tensor-core decode kernel for up to 8 tokens in one pass when the
// shape allows it (u4/u8 at group 64, K a multiple of 512, so a row's scales
// are whole 16-byte units for the bulk copies; 16-byte aligned weights).
// Rows of up to 5120 inputs run on one CTA each; longer rows of a plain
// u8 projection on a cluster of KS CTAs along K, the smallest KS for which
// K / KS is a multiple of 512 and at most 5120.  (For u4 the cluster kernel
// is faster on its own, 28.4 against 40.6 us for the 13824-input down
// projection at 8 tokens, but in a layer's kernel sequence the two 4-token
// streaming passes finish the layer sooner: the 48-layer stack takes 4.79
// ms with them and 4.99 ms with the split; for u8 the split wins both
// ways.)  *used tells the caller whether it ran.
cudaError_t launch_mma(int mode, const DenseParams &p, cudaStream_t st, bool *used) {
    *used = false;
    if (p.M < 2 || p.M > kMmaTokens || (p.bits != 4 && p.bits != 8) ||
        p.group != kGroup || p.K % 512 != 0 || !mma_aligned16(p.wq) ||
        !mma_aligned16(p.sc) || !mma_aligned16(p.bi))
        return cudaSuccess;
    constexpr int kMaxK = kGroup * kMmaGroupsPerWarp * kMmaMaxWarps;
    if (p.K > kMaxK) {
        if (mode != kMPlain || p.bits != 8) return cudaSuccess;
        int ks = 2;
        while (ks <= kMmaMaxSplit && (p.K % (512 * ks) != 0 || p.K / ks > kMaxK)) ++ks;
        if (ks > kMmaMaxSplit) return cudaSuccess;
#define GWA_MMA_SPLIT(B)                                                        \
    if (p.bits == B) {                                                          \
        if (ks == 2) return launch_mma_t<B, kMPlain, 2>(p, st, used);           \
        if (ks == 3) return launch_mma_t<B, kMPlain, 3>(p, st, used);           \
        return launch_mma_t<B, kMPlain, 4>(p, st, used);                        \
    }
        GWA_MMA_SPLIT(8)
#undef GWA_MMA_SPLIT
        return cudaSuccess;
    }
#define GWA_MMA_CASE(B)                                                            \
    if (p.bits == B) {                                                             \
        if (mode == kMPlain) return launch_mma_t<B, kMPlain, 1>(p, st, used);      \
        if (mode == kMSections) return launch_mma_t<B, kMSections, 1>(p, st, used); \
        if (mode == kMRope) return launch_mma_t<B, kMRope, 1>(p, st, used);        \
        return launch_mma_t<B, kMGateUp, 1>(p, st, used);                          \
    }
    GWA_MMA_CASE(4)
    GWA_MMA_CASE(8)
#undef GWA_MMA_CASE
    return cudaSuccess;
}

unsigned int mma_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_mma_timeouts, sizeof v);
    if (reset) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_mma_timeouts, &z, sizeof z);
    }
    return v;
}

}  // namespace gwa
