// Streaming decode kernel for one or two tokens, one quantization group per
// lane.  Same pipeline as qmv_stream.cu (a producer thread fills a
// shared-memory ring with whole packed rows and their scales and biases by
// bulk copy, consumer threads form exact integer dots), but each consumer
// lane owns a whole group of 64 inputs instead of a 16-byte chunk:
//  * the lane's activations of that group sit in 32 registers per token
//    (int16 pairs, one power-of-two scale per group, see common.cuh), so no
//    lane needs another lane's exponent;
//  * per row and group the lane reads 32 (u4) or 64 (u8) bytes of codes, one
//    scale and one bias, and applies the affine map once per group:
//      y += (s * 2^E) * D + b * sum_k x_k,   D = sum_k q_k * xi_k (exact);
//  * a row's groups are spread over 16-lane slices (ceil(G/16) slices per
//    row); each slice reduces its values with a 16-lane transpose reduction
//    and stores one partial per (row, token) in its own slot, and the
//    epilogue adds a row's slots in slice order (deterministic).
// Per 64 codes this costs one scale application and one reduction share
// instead of two, which is most of the non-dot work of the chunk layout.
// Sources: "Sanctum-MLX" (decode is a bandwidth-bound quantized GEMV); the
// packed format of "saragossa", "Quantization formats"; the fused QKV and
// gate+up epilogues of "The Cathedral Doubled Itself", "The two fusions".
#include "common.cuh"
#include "internal.h"

namespace gwa {

static __device__ unsigned int g_group_timeouts;

enum GroupMode { kGPlain = 0, kGSections = 1, kGGateUp = 2 };

constexpr int kSlice = 16;  // lanes per reduction slice
// Two CTAs per SM (this one and the next kernel's) must fit in registers.
constexpr int kGroupMaxThreads = 352;
// Shared memory per CTA: two CTAs (228 KB per SM, 1 KB reserved each).
constexpr size_t kGroupSmemCap = 110 * 1024;

// Activations of one group for MT tokens, encoded for the integer dot.
template <int MT>
struct GroupX {
    uint32_t pr[MT][32];  // int16 pairs in dp2a order
    float f[MT];          // 2^E (u4: 2^E / 16, see below)
    float xs[MT];         // plain fp32 sum of the group's activations
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

// Shared-memory image of the encoded activations, chunk-major so that the
// lanes of a warp (consecutive groups) read consecutive 16-byte chunks:
//   pairs[m][c][g] (uint4: pairs 4c..4c+3 of group g), then f[m][g],
//   xs[m][g].
template <int MT>
__host__ __device__ constexpr size_t xenc_bytes(int G) {
    return (size_t)MT * G * (8 * 16 + 8);
}

// All consumer threads encode x once per CTA: item (g, quarter) handles
// 16 inputs of group g; the four quarters of a group sit in four adjacent
// lanes and agree on the group's exponent and sum through shuffles.  A
// thread issues the loads of up to kXBatch items before encoding any, so
// long rows cost one memory round trip, not one per item.
constexpr int kXBatch = 4;

template <int BITS>
__device__ __forceinline__ void encode_quarter(const uint32_t (&u)[8], int it,
                                               int nq, int G, int m,
                                               uint4 *pairs, float *xf,
                                               float *xsm) {
    const int g = it >> 2, q = it & 3;
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
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
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
    if (it < nq) {
        pairs[((size_t)m * 8 + 2 * q) * G + g] =
            make_uint4(pr[0], pr[1], pr[2], pr[3]);
        pairs[((size_t)m * 8 + 2 * q + 1) * G + g] =
            make_uint4(pr[4], pr[5], pr[6], pr[7]);
        if (q == 0) {
            xf[(size_t)m * G + g] = BITS == 4 ? f * 0.0625f : f;
            xsm[(size_t)m * G + g] = sum;
        }
    }
}

template <int BITS, int MT>
__device__ __forceinline__ void encode_x_shared(const uint16_t *__restrict__ x,
                                                int M, int K, int G, int tid,
                                                int ncons,
                                                unsigned char *xenc) {
    uint4 *pairs = reinterpret_cast<uint4 *>(xenc);
    float *xf = reinterpret_cast<float *>(pairs + (size_t)MT * 8 * G);
    float *xsm = xf + (size_t)MT * G;
    const int nq = 4 * G;
    const int iters = (nq + ncons - 1) / ncons;  // same for every thread
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        for (int b0 = 0; b0 < iters; b0 += kXBatch) {
            uint32_t u[kXBatch][8];
#pragma unroll
            for (int j = 0; j < kXBatch; ++j) {
                const int it = (b0 + j) * ncons + tid;
                if (b0 + j < iters && it < nq && m < M) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        x + (int64_t)m * K + (int64_t)(it >> 2) * kGroup +
                        (it & 3) * 16);
                    const uint4 a = src[0], b = src[1];
                    u[j][0] = a.x; u[j][1] = a.y; u[j][2] = a.z; u[j][3] = a.w;
                    u[j][4] = b.x; u[j][5] = b.y; u[j][6] = b.z; u[j][7] = b.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) u[j][i] = 0u;
                }
            }
#pragma unroll
            for (int j = 0; j < kXBatch; ++j)
                if (b0 + j < iters)  // uniform: the shuffles need every lane
                    encode_quarter<BITS>(u[j], (b0 + j) * ncons + tid, nq, G,
                                         m, pairs, xf, xsm);
        }
    }
}

// A lane's group from the shared image (zeros for lanes without a group).
template <int MT>
__device__ __forceinline__ void load_group_x(const unsigned char *xenc, int G,
                                             int g, bool active,
                                             GroupX<MT> &gx) {
    const uint4 *pairs = reinterpret_cast<const uint4 *>(xenc);
    const float *xf = reinterpret_cast<const float *>(pairs + (size_t)MT * 8 * G);
    const float *xsm = xf + (size_t)MT * G;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 t = pairs[((size_t)m * 8 + c) * G + g];
            gx.pr[m][4 * c] = t.x;
            gx.pr[m][4 * c + 1] = t.y;
            gx.pr[m][4 * c + 2] = t.z;
            gx.pr[m][4 * c + 3] = t.w;
        }
        gx.f[m] = active ? xf[(size_t)m * G + g] : 0.f;
        gx.xs[m] = active ? xsm[(size_t)m * G + g] : 0.f;
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

// Transpose reduction of V values across the 16 lanes of a slice (the two
// halves of a warp reduce independently).  Afterwards slice lane l holds the
// slice sum of value index l >> (4 - log2 V); lanes whose low (4 - log2 V)
// bits are zero hold each index once.
template <int V>
__device__ __forceinline__ float slice_reduce(float (&v)[V], int lane) {
    static_assert(V >= 1 && V <= 16 && (V & (V - 1)) == 0, "V");
#pragma unroll
    for (int half = V / 2, bit = 8; half >= 1; half /= 2, bit /= 2) {
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
    for (int bit = 8 / V; bit >= 1; bit /= 2)
        r += __shfl_xor_sync(0xffffffffu, r, bit);
    return r;
}

__device__ __forceinline__ float slot_total(const float *red, int idx,
                                            int slices) {
    float t = 0.f;
    for (int s = 0; s < slices; ++s) t += red[idx * slices + s];
    return t;
}

// A stage holds UPS = RS * UPT units (rows, or gate/up row pairs).  Consumer
// half-warp h belongs to row group h / slices and covers groups
// [16 * (h % slices), +16) of that row group's RPH rows.  Half-warps past
// RS * slices (an odd count rounded up to whole warps) only take part in
// the shuffles.
template <int BITS, int MT, int MODE, int RPH>
__global__ void __maxnreg__(88)
    qmv_group_kernel(DenseParams p, int stages, int64_t units, int rs,
                     int slices, uint32_t xenc_off) {
    constexpr int HALVES = MODE == kGGateUp ? 2 : 1;
    constexpr int UPT = RPH / HALVES;
    constexpr int V = RPH * MT;
    constexpr int GB = BITS * 8;  // bytes of codes per row and group
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int ncons = blockDim.x - kWarp;
    const int lane = tid & (kWarp - 1);
    const int ups = rs * UPT;
    const uint32_t rowbytes = (uint32_t)p.K * BITS / 8;
    const uint32_t sbrow = (uint32_t)p.G * 2;
    const uint32_t rows_stage = (uint32_t)(HALVES * ups);
    const uint32_t stage_bytes = rows_stage * (rowbytes + 2 * sbrow);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    uint64_t *empty = full + stages;
    float *red = reinterpret_cast<float *>(empty + stages);
    __shared__ int s_issued, s_consumed;

    const int64_t u0 = units * blockIdx.x / gridDim.x;
    const int64_t u1 = units * (blockIdx.x + 1) / gridDim.x;
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
                    atomicAdd(&g_group_timeouts, 1u);
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
                    const int64_t r = ua + (h ? p.I : 0);
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
        const int hw = tid / kSlice;              // half-warp
        const bool in_group = hw < rs * slices;
        const int hg = in_group ? hw / slices : 0;  // row group
        const int sl = in_group ? hw - hg * slices : 0;
        const int g = sl * kSlice + (tid & (kSlice - 1));
        const bool active = in_group && g < p.G;
        // lanes without a group read group 0 (finite weights) with zero
        // activations, so their values are exact zeros
        const int gg = active ? g : 0;
        unsigned char *xenc = smem + xenc_off;
        pdl_wait_primary();  // x may be the previous kernel's output
        encode_x_shared<BITS, MT>(p.x, p.M, p.K, p.G, tid, ncons, xenc);
        // the consumer warps only (the producer is in its copy loop)
        asm volatile("bar.sync 1, %0;" ::"r"(ncons) : "memory");
        GroupX<MT> gx;
        load_group_x<MT>(xenc, p.G, gg, active, gx);
        uint32_t offw[RPH], offs[RPH];
        const uint32_t sb_delta = rows_stage * (uint32_t)p.G * 2u;
#pragma unroll
        for (int j = 0; j < RPH; ++j) {
            const uint32_t srow =
                (uint32_t)((j / UPT) * ups + hg * UPT + (j % UPT));
            offw[j] = srow * rowbytes + (uint32_t)gg * GB;
            offs[j] = rows_stage * rowbytes + (srow * (uint32_t)p.G + gg) * 2u;
        }
        for (int st = 0; st < nst; ++st) {
            const int s = st % stages;
            if (!mbar_wait(&full[s], (st / stages) & 1)) {
                atomicAdd(&g_group_timeouts, 1u);
                atomicMin(&s_consumed, st);
                break;
            }
            const int64_t ua = u0 + (int64_t)st * ups;
            const int n = (int)min((int64_t)ups, u1 - ua);
            const unsigned char *base = smem + (uint32_t)s * stage_bytes;
            float v[V];
#pragma unroll
            for (int j = 0; j < RPH; ++j) {
                uint4 w[BITS / 2];
#pragma unroll
                for (int i = 0; i < BITS / 2; ++i)
                    w[i] = reinterpret_cast<const uint4 *>(base + offw[j])[i];
                const float sv = bf16_bits_to_f32(
                    *reinterpret_cast<const uint16_t *>(base + offs[j]));
                const float bv = bf16_bits_to_f32(
                    *reinterpret_cast<const uint16_t *>(base + offs[j] +
                                                        sb_delta));
                int d[MT];
                group_dot<BITS, MT>(w, gx, d);
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    v[j * MT + m] =
                        fmaf(sv * gx.f[m], (float)d[m], bv * gx.xs[m]);
            }
            // every lane's reads of this stage are done: release the slot
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const float tot = slice_reduce<V>(v, lane);
            constexpr int SPREAD = kSlice / V;
            if (in_group && (lane & (SPREAD - 1)) == 0) {
                const int idx = (lane & (kSlice - 1)) / SPREAD;  // j*MT + m
                const int j = idx / MT, m = idx % MT;
                const int u = hg * UPT + (j % UPT), h = j / UPT;
                if (u < n)
                    red[((((st * ups + u) * HALVES + h) * MT + m) * slices) +
                        sl] = tot;
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
    for (int i = tid; i < nu * MT; i += blockDim.x) {
        const int lu = i / MT, m = i % MT;
        if (m >= p.M) continue;
        const int64_t n = u0 + lu;
        if constexpr (MODE == kGGateUp) {
            const float gv = slot_total(red, (lu * 2 + 0) * MT + m, slices);
            const float uv = slot_total(red, (lu * 2 + 1) * MT + m, slices);
            p.y[(int64_t)m * p.I + n] =
                f32_to_bf16_bits(gv / (1.0f + __expf(-gv)) * uv);
        } else if constexpr (MODE == kGPlain) {
            p.y[(int64_t)m * p.N + n] =
                f32_to_bf16_bits(slot_total(red, lu * MT + m, slices));
        } else {
            int s = 0;
            while (s + 1 < p.nsec && n >= p.sec_start[s + 1]) ++s;
            const int64_t j = n - p.sec_start[s];
            const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
            float val = slot_total(red, lu * MT + m, slices);
            if (p.sec_bias[s]) val += bf16_bits_to_f32(p.sec_bias[s][j]);
            p.sec_out[s][(int64_t)m * size + j] = f32_to_bf16_bits(val);
        }
    }
}

// ------------------------------------------------------------ host side
template <int BITS, int MT, int MODE, int RPH>
static cudaError_t launch_group_r(const DenseParams &p, cudaStream_t st,
                                  bool *used) {
    constexpr int HALVES = MODE == kGGateUp ? 2 : 1;
    constexpr int UPT = RPH / HALVES;
    const int64_t units = MODE == kGGateUp ? p.I : p.N;
    const size_t rowbytes = (size_t)p.K * BITS / 8;
    const size_t sbrow = (size_t)p.G * 2;
    const int slices = (p.G + kSlice - 1) / kSlice;
    // row groups: as many as fit the thread limit with the producer warp
    int rs = 1;
    while (rs < 8 && 2 * rs * slices * kSlice <= kGroupMaxThreads - kWarp)
        rs *= 2;
    const int ncons = ((rs * slices * kSlice + kWarp - 1) / kWarp) * kWarp;
    const int threads = ncons + kWarp;
    if (threads > kGroupMaxThreads) return cudaSuccess;  // not used
    const size_t stage_bytes = (size_t)HALVES * rs * UPT * (rowbytes + 2 * sbrow);
    // one CTA per SM, so the next kernel's CTA fits beside it and can
    // prefetch while this one drains
    int grid = num_sms();
    if ((int64_t)grid > units) grid = (int)units;
    const size_t red_bytes =
        (size_t)((units + grid - 1) / grid) * HALVES * MT * 4 * slices;
    const size_t fixed = 16 * 8 + ((red_bytes + 15) / 16) * 16 +
                         xenc_bytes<MT>(p.G);
    if (fixed >= kGroupSmemCap) return cudaSuccess;
    int stages = (int)((kGroupSmemCap - fixed) / stage_bytes);
    if (stages > 8) stages = 8;
    if (stages < 2) return cudaSuccess;  // rows too long for the ring
    const size_t xenc_off =
        stages * stage_bytes + 16 * stages + ((red_bytes + 15) / 16) * 16;
    const size_t smem = xenc_off + xenc_bytes<MT>(p.G);
    auto kern = qmv_group_kernel<BITS, MT, MODE, RPH>;
    int dummy = 0;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   threads, smem, &dummy);
    if (e != cudaSuccess) return e;
    *used = true;
    return launch_pdl(reinterpret_cast<const void *>(kern), grid, threads,
                      smem, st, p, stages, units, rs, slices,
                      (uint32_t)xenc_off);
}

static bool aligned16g(const void *q) {
    return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
}

// Launches the group-per-lane kernel when the shape allows it (one token,
// row strides of scales multiple of 16 bytes, 16-byte aligned bases);
// *used tells the caller whether it ran.
cudaError_t launch_group(int mode, const DenseParams &p, cudaStream_t st,
                         bool *used) {
    *used = false;
    if (p.M != 1 || (p.G % 8) != 0 || !aligned16g(p.sc) ||
        !aligned16g(p.bi) || !aligned16g(p.wq))
        return cudaSuccess;
    if (p.bits == 4) {
        if (mode == kGPlain) return launch_group_r<4, 1, kGPlain, 2>(p, st, used);
        if (mode == kGSections)
            return launch_group_r<4, 1, kGSections, 2>(p, st, used);
        return launch_group_r<4, 1, kGGateUp, 2>(p, st, used);
    }
    if (mode == kGPlain) return launch_group_r<8, 1, kGPlain, 2>(p, st, used);
    if (mode == kGSections)
        return launch_group_r<8, 1, kGSections, 2>(p, st, used);
    return launch_group_r<8, 1, kGGateUp, 2>(p, st, used);
}

unsigned int group_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_group_timeouts, sizeof v);
    if (reset) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_group_timeouts, &z, sizeof z);
    }
    return v;
}

}  // namespace gwa
