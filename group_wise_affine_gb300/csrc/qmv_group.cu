// Streaming decode kernel for one token, one 64-input chunk per lane.  Same
// pipeline as qmv_stream.cu (a producer thread fills a shared-memory ring
// with whole packed rows and their scales and biases by bulk copy, consumer
// threads form exact integer dots), but each consumer lane owns a chunk of
// 64 inputs (a group of 64, half a group of 128 or two groups of 32)
// instead of a 16-byte piece:
//  * the lane's activations of that chunk sit in 32 registers per token
//    (int16 pairs, one power-of-two scale per chunk, see common.cuh), so no
//    lane needs another lane's exponent;
//  * per row and chunk the lane reads 32 (u4) or 64 (u8) bytes of codes and
//    the scale and bias of each group the chunk covers, and applies the
//    affine map once per group:
//      y += (s * 2^E) * D + b * sum_k x_k,   D = sum_k q_k * xi_k (exact);
//  * a row's chunks are spread over 16-lane slices (ceil(K/64/16) slices
//    per row); each slice reduces its values with a 16-lane transpose
//    reduction and stores one partial per (row, token) in its own slot, and
//    the epilogue adds a row's slots in slice order (deterministic).
// Per 64 codes this costs one or two scale applications and one reduction
// share, against two of each in the 16-byte-piece layout.
//  * activations the int16 encoding would round by more than 2^-16 of a
//    group's magnitude (common.cuh, "marked groups") switch the whole CTA
//    (every CTA encodes the same activations) to a copy of the loop that
//    adds an int8 residual plane per chunk: about 40% more instructions per
//    row, taken only for such inputs.
//  * plain projections run as one-section calls of the sections kernel, so
//    a decoder layer's calls share two kernels' code in the SM's
//    instruction cache instead of three.
// Sources: "Sanctum-MLX" (decode is a bandwidth-bound quantized GEMV); the
// packed format of "saragossa", "Quantization formats"; the fused QKV and
// gate+up epilogues of "The Cathedral Doubled Itself", "The two fusions".
#include "group_dot.cuh"
#include "internal.h"

namespace gwa {

static __device__ unsigned int g_group_timeouts;

// Modes as the host passes them; a plain projection runs as one section.
enum GroupMode { kGPlain = 0, kGSections = 1, kGGateUp = 2, kGRope = 3 };

// QKV with the rotary embedding (kGRope): a unit is the pair of rows
// (i, i + d/2) of a head (rope_pair_row), cut into stages of whole pairs
// within one head.

constexpr int kSlice = 16;  // lanes per reduction slice
// Two CTAs per SM (this one and the next kernel's) must fit in registers:
// an SM's warps are spread over its four schedulers, each with a quarter of
// the register file (16K), so two CTAs of 11 warps put 6 warps on some
// scheduler and can use 80 registers a thread at most (88 would need 16896).
// The u4 loops fit in 80; the u8 ones keep 88 and take at most 9 warps a
// CTA instead (two CTAs of 9 warps put 5 on a scheduler: 14080 registers).
constexpr int kGroupMaxThreads = 352;
constexpr int kGroupMaxThreadsU8 = 288;
// Shared memory per CTA: two CTAs (228 KB per SM, 1 KB reserved each).
constexpr size_t kGroupSmemCap = 110 * 1024;

__device__ __forceinline__ float slot_total(const float *red, int idx,
                                            int slices) {
    float t = 0.f;
    for (int s = 0; s < slices; ++s) t += red[idx * slices + s];
    return t;
}

// The consumer side of the stage loop (see qmv_group_kernel), for a lane
// whose image is ready.  EX (two-plane path, common.cuh "marked groups"):
// once every lane holds its int16 pairs in registers, the image's pairs are
// dead, and all consumer threads write the chunks' int8 residual planes
// over them (group_plane_store); every row then takes both planes' dots in
// one pass over its code bytes.  The kernel has no local memory and no
// calls: a stack frame costs the SM the shared-memory carveout that lets
// two of these CTAs share it.
template <int BITS, int MT, int MODE, int RPH, int GS, bool EX>
__device__ __forceinline__ void group_loop(
    const uint16_t *x, int K, int G, unsigned char *smem, uint64_t *full,
    uint64_t *empty, float *red, int *s_consumed, int stages, int nst, int nu,
    int ups, int slices, uint32_t stage_bytes, uint32_t codes_off,
    uint32_t rows_stage, uint32_t rowbytes, int ncons, int tid,
    uint32_t xenc_off) {
    constexpr int HALVES = (MODE == kGGateUp || MODE == kGRope) ? 2 : 1;
    constexpr int UPT = RPH / HALVES;
    constexpr int V = RPH * MT;
    constexpr int GB = BITS * 8;  // bytes of codes per row and chunk
    constexpr bool SPLIT = GS == 32;
    const int lane = tid & (kWarp - 1);
    const int hw = tid / kSlice;  // half-warp
    const bool in_group = hw < ups / UPT * slices;  // row groups x slices
    const int hg = in_group ? hw / slices : 0;  // row group
    const int sl = in_group ? hw - hg * slices : 0;
    const int nchunk = K / 64;
    const int g = sl * kSlice + (tid & (kSlice - 1));  // chunk
    const bool active = in_group && g < nchunk;
    // lanes without a chunk read chunk 0 (finite weights) with zero
    // activations, so their values are exact zeros
    const int gg = active ? g : 0;
    // first weight group of the chunk
    const int sg = GS == 64 ? gg : GS == 128 ? gg >> 1 : 2 * gg;
    unsigned char *xenc = smem + xenc_off;
    GroupX<MT> gx;
    const int rot = chunk_rot<BITS>(gg);
    load_group_rows<MT, SPLIT>(xenc, MT, nchunk, 0, gg, active, gx,
                               image_shift<BITS>(gg));
    const uint4 *const plane = reinterpret_cast<const uint4 *>(xenc) + gg;
    static_assert(!EX || MT == 1, "two-plane path: one token");
    if constexpr (EX) {
        asm volatile("bar.sync 1, %0;" ::"r"(ncons) : "memory");
        group_plane_store<BITS>(x, K, 1, nchunk, nullptr, tid, ncons, xenc,
                                reinterpret_cast<uint4 *>(xenc));
        asm volatile("bar.sync 1, %0;" ::"r"(ncons) : "memory");
    }
    // the lane's reads of stage row srow(j) = (j / UPT) ups + hg UPT + j % UPT
    // (row j of its row group): codes at offw + srow(j) rowbytes, scale at
    // offs + 2 srow(j) G; rows past the end of a stage of fewer units read
    // the stage's first row instead (their values are never stored), so
    // that no read leaves a short slot
    // (the one-plane copy keeps each row's two offsets in registers; the
    // two-plane copy, short of registers, forms them per stage)
    const uint32_t sb_delta = rows_stage * (uint32_t)G * 2u;
    const uint32_t offw = codes_off + (uint32_t)gg * GB;
    const uint32_t offs = (uint32_t)sg * 2u;
    constexpr int NO = EX ? 1 : RPH;
    uint32_t offw_j[NO], offs_j[NO];
#pragma unroll
    for (int j = 0; j < NO; ++j) {
        const uint32_t srow = (uint32_t)((j / UPT) * ups + hg * UPT + (j % UPT));
        offw_j[j] = offw + srow * rowbytes;
        offs_j[j] = offs + srow * (uint32_t)G * 2u;
    }
    // this lane's slot of the partial sums: value index idx = j*MT + m
    // of unit u (stage-relative), half h
    constexpr int SPREAD = kSlice / V;
    const bool stores = in_group && (lane & (SPREAD - 1)) == 0;
    int lu, roff;
    {
        const int idx = (lane & (kSlice - 1)) / SPREAD;
        const int j = idx / MT, m = idx % MT;
        const int u = hg * UPT + (j % UPT), h = j / UPT;
        lu = u;
        roff = ((u * HALVES + h) * MT + m) * slices + sl;
    }
    const int rstep = ups * HALVES * MT * slices;
    int s = 0;
    uint32_t ph = 0;
    for (int st = 0; st < nst; ++st) {
        if (!mbar_wait(&full[s], ph)) {
            atomicAdd(&g_group_timeouts, 1u);
            atomicMin(s_consumed, st);
            break;
        }
        const unsigned char *base = smem + (uint32_t)s * stage_bytes;
        const int left = nu - st * ups;  // units in this stage: min(ups, left)
        float v[V];
#pragma unroll
        for (int j = 0; j < RPH; ++j) {
            const bool in = hg * UPT + (j % UPT) < left;
            uint32_t ow, os;
            if constexpr (EX) {
                const uint32_t srow =
                    in ? (uint32_t)((j / UPT) * ups + hg * UPT + (j % UPT)) : 0u;
                ow = offw + srow * rowbytes;
                os = offs + srow * (uint32_t)G * 2u;
            } else {
                ow = in ? offw_j[j] : offw;
                os = in ? offs_j[j] : offs;
            }
            uint4 w[BITS / 2];
            lds_group<BITS>(base + ow, rot, w);
            if constexpr (SPLIT) {
                // the scales and biases of the chunk's two groups
                const uint32_t s2 =
                    *reinterpret_cast<const uint32_t *>(base + os);
                const uint32_t b2 =
                    *reinterpret_cast<const uint32_t *>(base + os + sb_delta);
                int dl[MT], dh[MT], ll = 0, lh = 0;
                group_dot_split<BITS, MT>(w, gx, rot, dl, dh);
                if constexpr (EX)
                    group_dot_lo_split<BITS>(w, plane, nchunk, rot, ll, lh);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float fl = bf16_lo(s2) * gx.f[m];
                    const float fh = bf16_hi(s2) * gx.f[m];
                    float t = fmaf(bf16_lo(b2), gx.xs[m],
                                   bf16_hi(b2) * gx.xs2[m]);
                    if constexpr (EX)  // the residual plane, 2^-7 of the scale
                        t = fmaf(fl * 0.0078125f, (float)ll,
                                 fmaf(fh * 0.0078125f, (float)lh, t));
                    v[j * MT + m] =
                        fmaf(fl, (float)dl[m], fmaf(fh, (float)dh[m], t));
                }
            } else {
                const float sv = bf16_bits_to_f32(
                    *reinterpret_cast<const uint16_t *>(base + os));
                const float bv = bf16_bits_to_f32(
                    *reinterpret_cast<const uint16_t *>(base + os + sb_delta));
                int d[MT], dlo = 0;
                if constexpr (EX)
                    group_dot2<BITS, MT>(w, gx, plane, nchunk, d, dlo);
                else
                    group_dot<BITS, MT>(w, gx, d);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float sf = sv * gx.f[m];
                    float t = bv * gx.xs[m];
                    if constexpr (EX)  // the residual plane, 2^-7 of the scale
                        t = fmaf(sf * 0.0078125f, (float)dlo, t);
                    v[j * MT + m] = fmaf(sf, (float)d[m], t);
                }
            }
        }
        // every lane's reads of this stage are done: release the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        const float tot = sub_reduce<kSlice, V>(v, lane);
        if (stores && lu < nu) red[roff] = tot;
        lu += ups;
        roff += rstep;
        if (++s == stages) {
            s = 0;
            ph ^= 1;
        }
    }
}

// A stage holds UPS = RS * UPT units (rows, or gate/up row pairs).  Consumer
// half-warp h belongs to row group h / slices and covers groups
// [16 * (h % slices), +16) of that row group's RPH rows.  Half-warps past
// RS * slices (an odd count rounded up to whole warps) only take part in
// the shuffles.
template <int BITS, int MT, int MODE, int RPH, int GS>
__global__ void __maxnreg__(BITS == 4 ? 80 : 88)
    qmv_group_kernel(DenseParams p, int stages, int64_t units, int rs,
                     int slices, uint32_t ring_bytes, uint32_t xenc_off,
                     uint32_t rope_off) {
    constexpr int HALVES = (MODE == kGGateUp || MODE == kGRope) ? 2 : 1;
    constexpr int UPT = RPH / HALVES;
    constexpr int V = RPH * MT;
    constexpr int GB = BITS * 8;  // bytes of codes per row and chunk
    constexpr bool SPLIT = GS == 32;  // a chunk covers two groups
    extern __shared__ __align__(128) unsigned char smem[];

    const int tid = threadIdx.x;
    const int ncons = blockDim.x - kWarp;
    const int lane = tid & (kWarp - 1);
    const int ups = rs * UPT;
    const uint32_t rowbytes = (uint32_t)p.K * BITS / 8;
    const uint32_t sbrow = (uint32_t)p.G * 2;
    const uint32_t rows_stage = (uint32_t)(HALVES * ups);
    const uint32_t stage_bytes = rows_stage * (rowbytes + 2 * sbrow);
    // A stage holds its rows' scales, then their biases, then their codes,
    // so a stage of fewer units needs only a prefix of the slot: the last
    // slot of the ring may be such a short one (see the host side).
    const uint32_t codes_off = 2 * rows_stage * sbrow;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + ring_bytes);
    uint64_t *empty = full + stages;
    float *red = reinterpret_cast<float *>(empty + stages);
    __shared__ int s_issued, s_consumed;
    __shared__ int s_marked;  // the encode met a marked chunk

    // rope: whole stages per CTA (ups divides d/2), so no stage crosses a head
    const int64_t ualign = MODE == kGRope ? rs * UPT : 1;
    const int64_t u0 = units / ualign * blockIdx.x / gridDim.x * ualign;
    const int64_t u1 = units / ualign * (blockIdx.x + 1) / gridDim.x * ualign;
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
        s_marked = 0;
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
            int s = 0;        // ring slot of stage st
            uint32_t ph = 0;  // its use count parity
            for (int st = 0; st < nst; ++st) {
                // Weights are never written by this library's kernels, and a
                // kernel of any other kind completes before one of ours starts
                // (it never triggers an early launch), so the first `stages`
                // stages can be fetched before the previous grid finishes.
                if (st == stages) pdl_wait_primary();
                if (st >= stages && !mbar_wait(&empty[s], ph ^ 1)) {
                    atomicAdd(&g_group_timeouts, 1u);
                    break;
                }
                const int64_t ua = u0 + (int64_t)st * ups;
                const int n = (int)min((int64_t)ups, u1 - ua);
                unsigned char *base = smem + (size_t)s * stage_bytes;
                unsigned char *dsc = base;
                unsigned char *dbi = dsc + rows_stage * sbrow;
                unsigned char *dwq = base + codes_off;
                mbar_expect_tx(&full[s], (uint32_t)(HALVES * n) *
                                             (rowbytes + 2 * sbrow));
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    const int64_t r = MODE == kGRope ? rope_pair_row(ua, h, p.rope_hd)
                                                     : ua + (h ? p.I : 0);
                    bulk_g2s(dwq + h * ups * rowbytes, wq + r * rowbytes,
                             n * rowbytes, &full[s]);
                    bulk_g2s(dsc + h * ups * sbrow, sc + r * sbrow, n * sbrow,
                             &full[s]);
                    bulk_g2s(dbi + h * ups * sbrow, bi + r * sbrow, n * sbrow,
                             &full[s]);
                }
                s_issued = st + 1;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
    } else {
        // ------------------------------------------------ consumers
        // (the lane layout is group_loop's: chunk g of row group hg)
        const int hw = tid / kSlice;              // half-warp
        const bool in_group = hw < rs * slices;
        const int hg = in_group ? hw / slices : 0;  // row group
        const int sl = in_group ? hw - hg * slices : 0;
        const int nchunk = p.K / 64;
        const int g = sl * kSlice + (tid & (kSlice - 1));  // chunk
        const bool active = in_group && g < nchunk;
        const int gg = active ? g : 0;
        unsigned char *xenc = smem + xenc_off;
        if constexpr (MODE == kGRope) {
            // the CTA's (cos, sin) table, while the previous kernel drains
            // (positions are an input no kernel of this library writes); it
            // is read in the epilogue, after the block barrier
            float2 *cs = reinterpret_cast<float2 *>(smem + rope_off);
            const int half = p.rope_hd / 2;
            for (int e = tid; e < nu * MT; e += ncons) {
                const int64_t n = u0 + e / MT;
                if (rope_pair_row(n, 0, p.rope_hd) < p.rope_end)
                    cs[e] = rope_cos_sin(p.rope_pos[e % MT], (int)(n % half),
                                         p.rope_r);
            }
        }
        pdl_wait_primary();  // x may be the previous kernel's output
        encode_rows_shared<BITS, SPLIT, kMarkDefer>(p.x, p.M, MT, p.K, nchunk,
                                                    tid, ncons, xenc, nullptr,
                                                    &s_marked);
        // the consumer warps only (the producer is in its copy loop)
        asm volatile("bar.sync 1, %0;" ::"r"(ncons) : "memory");
        // Marked chunks (common.cuh, "marked groups"): if the encode flagged
        // one, the CTA runs the two-plane loop (every CTA encodes the same
        // activations, so all decide alike).
        if (s_marked)
            group_loop<BITS, MT, MODE, RPH, GS, true>(
                p.x, p.K, p.G, smem, full, empty, red, &s_consumed, stages, nst,
                nu, ups, slices, stage_bytes, codes_off, rows_stage, rowbytes,
                ncons, tid, xenc_off);
        else
            group_loop<BITS, MT, MODE, RPH, GS, false>(
                p.x, p.K, p.G, smem, full, empty, red, &s_consumed, stages, nst,
                nu, ups, slices, stage_bytes, codes_off, rows_stage, rowbytes,
                ncons, tid, xenc_off);
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
        } else if constexpr (MODE == kGRope) {
            // pair (r0, r0 + d/2) of a head; sections are whole heads
            const int half = p.rope_hd / 2;
            float a = slot_total(red, (lu * 2 + 0) * MT + m, slices);
            float b = slot_total(red, (lu * 2 + 1) * MT + m, slices);
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
                const float2 c =
                    reinterpret_cast<const float2 *>(smem + rope_off)[i];
                const float a2 = a * c.x - b * c.y;
                b = b * c.x + a * c.y;
                a = a2;
            }
            uint16_t *o = p.sec_out[s] + (int64_t)m * size + j;
            o[0] = f32_to_bf16_bits(a);
            o[half] = f32_to_bf16_bits(b);
        } else if (p.nsec == 1) {
            // a plain projection: no section lookup
            const float val = slot_total(red, lu * MT + m, slices);
            p.sec_out[0][(int64_t)m * p.N + n] = f32_to_bf16_bits(
                p.sec_bias[0] ? val + bf16_bits_to_f32(p.sec_bias[0][n]) : val);
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
template <int BITS, int MT, int MODE, int RPH, int GS>
static cudaError_t launch_group_r(const DenseParams &p, cudaStream_t st,
                                  bool *used) {
    constexpr int HALVES = (MODE == kGGateUp || MODE == kGRope) ? 2 : 1;
    constexpr int UPT = RPH / HALVES;
    const int64_t units =
        MODE == kGGateUp ? p.I : MODE == kGRope ? p.N / 2 : p.N;
    const size_t rowbytes = (size_t)p.K * BITS / 8;
    const size_t sbrow = (size_t)p.G * 2;
    const int nchunk = p.K / 64;
    const int slices = (nchunk + kSlice - 1) / kSlice;
    // row groups: as many as fit the thread limit with the producer warp
    // (a power of two for the rotary mode, whose stages hold whole pairs of
    // a head)
    constexpr int kMax = BITS == 8 ? kGroupMaxThreadsU8 : kGroupMaxThreads;
    int rs = 1;
    if (MODE == kGRope) {
        while (rs < 8 && 2 * rs * slices * kSlice <= kMax - kWarp) rs *= 2;
    } else {
        rs = (kMax - kWarp) / (slices * kSlice);
        rs = rs < 1 ? 1 : rs > 8 ? 8 : rs;
    }
    const int ncons = ((rs * slices * kSlice + kWarp - 1) / kWarp) * kWarp;
    const int threads = ncons + kWarp;
    if (threads > kMax) return cudaSuccess;  // not used
    // rope: stages of whole pairs within one head
    if (MODE == kGRope && ((p.rope_hd / 2) % (rs * UPT)) != 0)
        return cudaSuccess;  // not used
    const size_t stage_bytes = (size_t)HALVES * rs * UPT * (rowbytes + 2 * sbrow);
    // one CTA per SM, so the next kernel's CTA fits beside it and can
    // prefetch while this one drains
    int grid = num_sms();
    if ((int64_t)grid > units) grid = (int)units;
    // units per CTA, at most (rope: plus one stage for the alignment)
    const int64_t umax = (units + grid - 1) / grid + (MODE == kGRope ? rs * UPT : 0);
    const size_t red_bytes = (size_t)umax * HALVES * MT * 4 * slices;
    // (cos, sin) per pair and token; rounded to 16 bytes, since the
    // activation image after it is read and written in 16-byte units
    const size_t rope_bytes =
        MODE == kGRope ? ((size_t)umax * MT * 8 + 15) / 16 * 16 : 0;
    const size_t fixed = 16 * 8 + ((red_bytes + 15) / 16) * 16 + rope_bytes +
                         ximg_bytes(MT, nchunk, GS == 32);
    if (fixed >= kGroupSmemCap) return cudaSuccess;
    int stages = (int)((kGroupSmemCap - fixed) / stage_bytes);
    if (stages > 8) stages = 8;
    if (stages < 2) return cudaSuccess;  // rows too long for the ring
    size_t ring = (size_t)stages * stage_bytes;
    // When every CTA's share is at most one stage more than the ring holds,
    // a short last slot (a prefix of a stage: scales, biases, then the codes
    // of the units it carries) can take that stage, so the whole share is
    // fetched before the previous kernel finishes and no fetch is left for
    // after the activations arrive.
    const int64_t ups = (int64_t)rs * UPT;
    if (stages < 8 && umax > stages * ups && umax <= (stages + 1) * ups) {
        const int64_t tail = umax - stages * ups;
        const size_t foot = (size_t)2 * HALVES * ups * sbrow +
                            (size_t)((HALVES - 1) * ups + tail) * rowbytes;
        if (fixed + ring + foot <= kGroupSmemCap) {
            ++stages;
            ring += foot;
        }
    }
    const size_t rope_off = ring + 16 * stages + ((red_bytes + 15) / 16) * 16;
    const size_t xenc_off = rope_off + rope_bytes;
    const size_t smem = xenc_off + ximg_bytes(MT, nchunk, GS == 32);
    auto kern = qmv_group_kernel<BITS, MT, MODE, RPH, GS>;
    int dummy = 0;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   threads, smem, &dummy);
    if (e != cudaSuccess) return e;
    *used = true;
    return launch_pdl(reinterpret_cast<const void *>(kern), grid, threads,
                      smem, st, p, stages, units, rs, slices, (uint32_t)ring,
                      (uint32_t)xenc_off, (uint32_t)rope_off);
}

static bool aligned16g(const void *q) {
    return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
}

template <int GS>
static cudaError_t launch_group_gs(int mode, const DenseParams &p,
                                   cudaStream_t st, bool *used) {
    if (mode == kGRope)
        return p.bits == 4 ? launch_group_r<4, 1, kGRope, 2, GS>(p, st, used)
                           : launch_group_r<8, 1, kGRope, 2, GS>(p, st, used);
    // A plain projection runs as one section: the same kernel as the fused
    // QKV projection, so that a layer's calls share their code (the SM's
    // instruction cache holds two of these kernels, not three).
    DenseParams q = p;
    if (mode == kGPlain) {
        q.nsec = 1;
        q.sec_start[0] = 0;
        q.sec_start[1] = p.N;
        q.sec_out[0] = p.y;
        q.sec_bias[0] = nullptr;
        mode = kGSections;
    }
    if (p.bits == 4) {
        if (mode == kGSections)
            return launch_group_r<4, 1, kGSections, 2, GS>(q, st, used);
        return launch_group_r<4, 1, kGGateUp, 2, GS>(q, st, used);
    }
    if (mode == kGSections)
        return launch_group_r<8, 1, kGSections, 2, GS>(q, st, used);
    return launch_group_r<8, 1, kGGateUp, 2, GS>(q, st, used);
}

// Launches the chunk-per-lane kernel when the shape allows it (one token,
// u4 or u8 codes in groups of 32, 64 or 128, whole 64-input chunks, row
// strides of scales multiple of 16 bytes, 16-byte aligned bases); *used
// tells the caller whether it ran.
cudaError_t launch_group(int mode, const DenseParams &p, cudaStream_t st,
                         bool *used) {
    *used = false;
    if (p.M != 1 || (p.bits != 4 && p.bits != 8) || (p.K % 64) != 0 ||
        (p.G % 8) != 0 || !aligned16g(p.sc) || !aligned16g(p.bi) ||
        !aligned16g(p.wq))
        return cudaSuccess;
    switch (p.group) {
        case 64: return launch_group_gs<64>(mode, p, st, used);
        case 32: return launch_group_gs<32>(mode, p, st, used);
        case 128: return launch_group_gs<128>(mode, p, st, used);
        default: return cudaSuccess;
    }
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
