// Streaming decode kernels (M <= 2): the weight rows a CTA owns are copied
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
#include "common.cuh"
#include "internal.h"

namespace gwa {

static __device__ unsigned int g_stream_timeouts;

enum StreamMode { kSPlain = 0, kSSections = 1, kSGateUp = 2 };

// A thread's activations for its chunk, encoded for the integer dot (see
// common.cuh): int16 pairs in dp2a order, the group scale 2^E and the plain
// fp32 sum of the chunk's activations.
template <int BITS, int MT>
struct XRegs {
    static constexpr int CODES = Fmt<BITS>::kChunkCodes;
    uint32_t pr[MT][CODES / 2];
    float f[MT];
    float xs[MT];
};

// Loads and encodes chunk c of each token.  Every lane of the warp must
// call this (the lanes of one group agree on its scale through shuffles);
// inactive lanes encode zeros.
template <int BITS, int MT>
__device__ __forceinline__ void load_x_regs(const uint16_t *__restrict__ x,
                                            int M, int K, int c, bool active,
                                            XRegs<BITS, MT> &xr) {
    constexpr int CODES = Fmt<BITS>::kChunkCodes;
    constexpr int CPG = kGroup / CODES;  // lanes sharing a group
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
        xr.xs[m] = xs;
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
                const uint32_t lo = word & 0x0f0f0f0fu;
                const uint32_t hi = (word >> 4) & 0x0f0f0f0fu;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t *pr = xr.pr[m] + 4 * wd;
                    int a = d[r][m][wd & 1];
                    a = dp2a_lo(pr[0], lo, a);
                    a = dp2a_hi(pr[1], lo, a);
                    a = dp2a_lo(pr[2], hi, a);
                    d[r][m][wd & 1] = dp2a_hi(pr[3], hi, a);
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
        for (int m = 0; m < MT; ++m)
            out[r][m] = fmaf(s[r] * xr.f[m], (float)(d[r][m][0] + d[r][m][1]),
                             b[r] * xr.xs[m]);
}

// RBU units per stage; a gate+up unit is one gate row plus one up row.
template <int BITS, int MT, int MODE, int RBU>
__global__ void __launch_bounds__(kStreamMaxThreads)
    qmv_stream_kernel(DenseParams p, int stages, int64_t units) {
    constexpr int HALVES = MODE == kSGateUp ? 2 : 1;
    constexpr int ROWS = HALVES * RBU;  // weight rows per stage
    constexpr int V = ROWS * MT;        // values reduced per warp per stage
    constexpr int RBATCH = MT == 1 ? 8 : 4;  // rows computed together
    constexpr int CODES = Fmt<BITS>::kChunkCodes;
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int ncons = blockDim.x - kWarp;
    const int lane = tid & (kWarp - 1);
    const uint32_t rowbytes = (uint32_t)p.K * BITS / 8;
    const uint32_t sbrow = (uint32_t)p.G * 2;
    const uint32_t stage_bytes = ROWS * (rowbytes + 2 * sbrow);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    uint64_t *empty = full + stages;
    float *red = reinterpret_cast<float *>(empty + stages);
    __shared__ int s_issued, s_consumed;

    const int64_t u0 = units * blockIdx.x / gridDim.x;
    const int64_t u1 = units * (blockIdx.x + 1) / gridDim.x;
    const int nu = (int)(u1 - u0);
    const int nst = (nu + RBU - 1) / RBU;

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], ncons / kWarp);
        }
        fence_mbar_init();
    }
    if (tid == 0) {
        s_issued = 0;
        s_consumed = nst;
        // let the next kernel in the stream start its own weight prefetch
        pdl_launch_dependents();
    }
    const int nwarps = ncons / kWarp;
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
                const int64_t ua = u0 + (int64_t)st * RBU;
                const int n = (int)min((int64_t)RBU, u1 - ua);
                unsigned char *base = smem + (size_t)s * stage_bytes;
                unsigned char *dcodes = base;
                unsigned char *dsc = base + ROWS * rowbytes;
                unsigned char *dbi = dsc + ROWS * sbrow;
                mbar_expect_tx(&full[s], (uint32_t)(HALVES * n) *
                                             (rowbytes + 2 * sbrow));
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    const int64_t r = ua + (h ? p.I : 0);
                    bulk_g2s(dcodes + h * RBU * rowbytes, wq + r * rowbytes,
                             n * rowbytes, &full[s]);
                    bulk_g2s(dsc + h * RBU * sbrow, sc + r * sbrow, n * sbrow,
                             &full[s]);
                    bulk_g2s(dbi + h * RBU * sbrow, bi + r * sbrow, n * sbrow,
                             &full[s]);
                }
                s_issued = st + 1;
            }
        }
    } else {
        // ------------------------------------------------ consumers
        const int c = tid;
        const bool active = c < p.nch;
        XRegs<BITS, MT> xr;
        pdl_wait_primary();  // x may be the previous kernel's output
        load_x_regs<BITS, MT>(p.x, p.M, p.K, c, active, xr);
        // lanes past the row end use chunk 0 (and its group) with zero
        // activations, so every value they read is a finite weight
        const int cc = active ? c : 0;
        const int g = (cc * CODES) / kGroup;
        for (int st = 0; st < nst; ++st) {
            const int s = st % stages;
            if (!mbar_wait(&full[s], (st / stages) & 1)) {
                atomicAdd(&g_stream_timeouts, 1u);
                atomicMin(&s_consumed, st);
                break;
            }
            const int64_t ua = u0 + (int64_t)st * RBU;
            const int n = (int)min((int64_t)RBU, u1 - ua);
            const unsigned char *base = smem + (size_t)s * stage_bytes;
            const uint16_t *ssc =
                reinterpret_cast<const uint16_t *>(base + ROWS * rowbytes);
            const uint16_t *sbi = ssc + ROWS * p.G;
            float v[V];
            // Rows are processed in batches with every load issued first and
            // no per-row branches, so the unpack/FMA chains of the rows in a
            // batch interleave.  Row slots past the stage end hold stale
            // data; their totals are dropped below.  Lanes past the row end
            // read chunk 0 with zero activations and contribute zero.
            const unsigned char *rowp = base + (size_t)cc * 16;
#pragma unroll
            for (int j0 = 0; j0 < ROWS; j0 += RBATCH) {
                uint4 w[RBATCH];
                float sv[RBATCH], bv[RBATCH];
#pragma unroll
                for (int jj = 0; jj < RBATCH; ++jj) {
                    const int j = j0 + jj;
                    w[jj] = *reinterpret_cast<const uint4 *>(
                        rowp + (size_t)j * rowbytes);
                    sv[jj] = bf16_bits_to_f32(ssc[j * p.G + g]);
                    bv[jj] = bf16_bits_to_f32(sbi[j * p.G + g]);
                }
                float o[RBATCH][MT];
                batch_dot<BITS, MT, RBATCH>(w, sv, bv, xr, o);
#pragma unroll
                for (int jj = 0; jj < RBATCH; ++jj)
#pragma unroll
                    for (int m = 0; m < MT; ++m) v[(j0 + jj) * MT + m] = o[jj][m];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const float tot = transpose_reduce<V>(v, lane);
            constexpr int SPREAD = kWarp / V;
            if ((lane & (SPREAD - 1)) == 0) {
                const int idx = lane / SPREAD;  // j * MT + m
                const int j = idx / MT, m = idx % MT;
                const int uj = j % RBU, h = j / RBU;
                // per-warp slot: the epilogue adds the warps in a fixed order
                if (uj < n)
                    red[(((st * RBU + uj) * HALVES + h) * MT + m) * nwarps +
                        tid / kWarp] = tot;
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
    auto total = [&](int idx) {
        float t = 0.f;
        for (int w = 0; w < nwarps; ++w) t += red[idx * nwarps + w];
        return t;
    };
    for (int i = tid; i < nu * MT; i += blockDim.x) {
        const int lu = i / MT, m = i % MT;
        if (m >= p.M) continue;
        const int64_t n = u0 + lu;
        if constexpr (MODE == kSGateUp) {
            const float gv = total((lu * 2 + 0) * MT + m);
            const float uv = total((lu * 2 + 1) * MT + m);
            p.y[(int64_t)m * p.I + n] = f32_to_bf16_bits(
                gv / (1.0f + __expf(-gv)) * uv);
        } else if constexpr (MODE == kSPlain) {
            p.y[(int64_t)m * p.N + n] = f32_to_bf16_bits(total(lu * MT + m));
        } else {
            int s = 0;
            while (s + 1 < p.nsec && n >= p.sec_start[s + 1]) ++s;
            const int64_t j = n - p.sec_start[s];
            const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
            float val = total(lu * MT + m);
            if (p.sec_bias[s]) val += bf16_bits_to_f32(p.sec_bias[s][j]);
            p.sec_out[s][(int64_t)m * size + j] = f32_to_bf16_bits(val);
        }
    }
}

// ------------------------------------------------------------ host side
template <int BITS, int MT, int MODE, int RBU>
static cudaError_t launch_stream_t(const DenseParams &p, cudaStream_t st,
                                   bool *used) {
    constexpr int HALVES = MODE == kSGateUp ? 2 : 1;
    const int64_t units = MODE == kSGateUp ? p.I : p.N;
    const size_t rowbytes = (size_t)p.K * BITS / 8;
    const size_t sbrow = (size_t)p.G * 2;
    const size_t stage_bytes = HALVES * RBU * (rowbytes + 2 * sbrow);
    int stages = (int)(kStreamRingTarget / stage_bytes);
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    const int ncons = ((p.nch + kWarp - 1) / kWarp) * kWarp;
    const int threads = ncons + kWarp;
    if (threads > kStreamMaxThreads) return cudaSuccess;  // not used
    auto kern = qmv_stream_kernel<BITS, MT, MODE, RBU>;
    // first pass: occupancy with a generous accumulator estimate
    const int sms = num_sms();
    const int nwarps = ncons / kWarp;
    size_t red_bytes =
        (size_t)((units + sms - 1) / sms + 1) * HALVES * MT * 4 * nwarps;
    size_t smem = stages * stage_bytes + 16 * stages + red_bytes;
    if (smem > kMaxDynSmem) return cudaSuccess;
    int grid = 0;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   threads, smem, &grid);
    if (e != cudaSuccess) return e;
    if ((int64_t)grid > units) grid = (int)units;
    red_bytes = (size_t)((units + grid - 1) / grid) * HALVES * MT * 4 * nwarps;
    smem = stages * stage_bytes + 16 * stages + red_bytes;
    *used = true;
    return launch_pdl(reinterpret_cast<const void *>(kern), grid, threads,
                      smem, st, p, stages, units);
}

static bool aligned16(const void *q) {
    return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
}

// Launches the streaming kernel when the shape allows it (M <= 2, row
// strides of scales multiple of 16 bytes, 16-byte aligned bases); *used
// tells the caller whether it ran.
cudaError_t launch_stream(int mode, const DenseParams &p, cudaStream_t st,
                          bool *used) {
    *used = false;
    if (p.M > 2 || (p.G % 8) != 0 || !aligned16(p.sc) || !aligned16(p.bi) ||
        !aligned16(p.wq))
        return cudaSuccess;
#define GWA_STREAM_CASE(B, MTV)                                              \
    if (p.bits == B && (MTV == 1 ? p.M == 1 : p.M == 2)) {                   \
        if (mode == kSPlain) return launch_stream_t<B, MTV, kSPlain, 8>(p, st, used); \
        if (mode == kSSections)                                              \
            return launch_stream_t<B, MTV, kSSections, 8>(p, st, used);      \
        return launch_stream_t<B, MTV, kSGateUp, 4>(p, st, used);            \
    }
    GWA_STREAM_CASE(4, 1)
    GWA_STREAM_CASE(4, 2)
    GWA_STREAM_CASE(8, 1)
    GWA_STREAM_CASE(8, 2)
#undef GWA_STREAM_CASE
    return cudaSuccess;
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
