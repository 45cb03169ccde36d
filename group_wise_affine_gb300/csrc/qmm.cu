// Prefill-shaped (M > 8) path on the 5th-generation tensor cores (tcgen05).
// "Sanctum-MLX", prefill paragraph: prefill is dominated by the matrix
// products of the quantized layers, so here the projection is a dense
// contraction.  Same operation as the decode path: y = x . (s*q + b)^T.
//
// Exact operands.  A bf16 scale times a centred 4-bit code, s*(q-8), has at
// most 8 + 3 significant bits and is exact in fp16 (for scales in fp16's
// normal range).  So each weight tile enters the MMA as fp16 s*(q-8) and the
// rest of the affine map goes into extra K columns:
//   s*q + b = s*(q-8) + b',   b' = b + 8s   (u4)
//   s*q + b = 16s*(qh-8) + s*(ql-8) + b',   b' = b + 136s   (u8, q = 16qh+ql)
//   y[m,n] = sum_k x[m,k] w'[n,k] + sum_g b'[n,g] X[m,g],  X = per-group sum.
// b' and X are split into fp16 hi + lo parts and the bias term is carried by
// three extra columns per group (b'hi*Xhi + b'hi*Xlo + b'lo*Xhi), laid out
// as three sections of G columns (Xhi | Xlo | Xhi against b'hi | b'hi |
// b'lo), so that 8 groups' columns come from one 16-byte load.  Activations
// are converted to fp16 once per call by a pre-pass; products are exact and
// accumulate in fp32 in tensor memory.
//
// Range.  fp16 covers 2^-14 .. 65504, bf16 2^-133 .. 3.4e38.  So every token
// and every weight row is scaled by a power of two before the conversion:
// token m by 2^e_m, which brings the largest of its |x| and of its group
// sums |X| into [2^14, 2^15) (pre-pass); row n by 2^f_n, which brings the
// largest of its |s| * 8 (u4; 128 for u8, the largest |16 s (qh-8)|) and
// |b'| there (dequantizers, once per tile).  The fp32 epilogue multiplies by
// 2^-f_n and 2^-e_m, both exact.  Values then stay exact wherever they lie
// within 2^24 of the largest of their token or row; smaller ones fall into
// fp16's subnormals and keep an error below 2^-25 of that largest, which is
// below the fp32 rounding of a sum that holds it.
//
// Kernel shape.  A CTA computes one 128-row weight tile (for gate+up: 64 gate
// rows and the matching 64 up rows) against NT = 16, 128 or 256 tokens, one
// MMA of M = 128, N = NT, K = 16 per 16 columns.  A K block's activation
// tile (shared memory) and A columns (tensor memory) share one ring slot, so
// the MMA issuer waits on one barrier and commits to one per K block; for
// 16 tokens, whose MMAs are short, a slot holds two K blocks (a lone
// issuing thread spends about as long on a wait or a commit as on an MMA,
// while at 128 or 256 tokens the coarser slots cost more in pipeline depth
// than they save):
//   warp 0    allocates tensor memory and, from one thread, loads with TMA
//             per 64-wide K block the activation tile (128-byte swizzle);
//   warp 1    issues tcgen05.mma (A from tensor memory, B from smem);
//   warp 2    loads, from one thread, the packed code tile of the 128 rows
//             per K block and per 8 K blocks the rows' scale tiles, which run
//             ahead as far as their own rings allow;
//   warps 3-18 dequantize: four warps per tensor-memory lane quarter take
//             every fourth K block, so each has four MMA periods for its
//             block; a thread turns its row's codes into fp16 pairs and
//             writes them to tensor memory with tcgen05.st (the A operand),
//             then reads the fp32 accumulators back with tcgen05.ld for the
//             epilogue (gate+up: the gate warps pass their values to the up
//             warps through shared memory).
// K split: when a projection's tiles leave SMs idle and fit one wave of
// clusters, the ks CTAs of a cluster share a tile, each taking a run of K
// blocks; ranks 1.. leave their fp32 partial sums in shared memory and rank
// 0 adds them through distributed shared memory before the epilogue
// (qmm_tc_kernel<..., true>).
// Every wait is bounded (2 s); a wait that runs out flags the workspace
// status word and the kernel unwinds without hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "cluster.cuh"
#include "common.cuh"
#include "qmm.h"

namespace gwa {

constexpr int kQmmDeqWarps = 16;     // four per tensor-memory lane quarter
constexpr int kQmmDeq0 = 3;          // first dequantizing warp
constexpr int kQmmThreads = (kQmmDeq0 + kQmmDeqWarps) * 32;
constexpr int kQmmRows = 128;        // weight rows per CTA (MMA M)
constexpr int kQmmSStages = 2;       // scale/bias-tile ring (8 K blocks each)
constexpr int kQmmMaxSplit = 4;      // CTAs per cluster splitting K
constexpr int kStatusBytes = 256;

// status word bit: a pipeline wait ran out
constexpr unsigned kStTimeout = 1u;

static __device__ unsigned int g_qmm_timeouts;

// K plus the bias columns, padded to whole pairs of 64-column K blocks (K
// itself is a multiple of 512), so a ring slot of two K blocks never holds
// a lone one.
static int64_t qmm_kext(int64_t K) {
    const int64_t G = K / 64;
    return K + ((3 * G + 127) / 128) * 128;
}

// Workspace: status word (256 bytes), the fp16 activations with their bias
// columns [M, kext], then each token's factor 2^-e_m [M] (fp32).
static size_t qmm_xe_bytes(int64_t M, int64_t K) {
    return (((size_t)M * (size_t)qmm_kext(K) * 2 + 255) / 256) * 256;
}

size_t qmm_workspace_bytes(int64_t M, int64_t K) {
    return kStatusBytes + qmm_xe_bytes(M, K) + (((size_t)M * 4 + 255) / 256) * 256;
}

// 2^p and 2^-p for the power p that brings t (> 0, finite) into
// [2^14, 2^15), with p clamped so that both stay normal fp32 numbers.
__device__ __forceinline__ void range_scale(float t, float &up, float &down) {
    int p = 0;
    if (t > 0.f && t < 3.0e38f) p = 141 - f32_exp_field(t);
    p = p < -125 ? -125 : p > 125 ? 125 : p;
    up = __uint_as_float((uint32_t)(127 + p) << 23);
    down = __uint_as_float((uint32_t)(127 - p) << 23);
}

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(dst_smem)),
        "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                     taddr),
                 "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
        "[%0];" ::"r"(smem_u32(bar))
        : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem]^T, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem,
                                          uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, "
        "%7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, "
        "%21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
          "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
          "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 4 consecutive 32-bit columns of this warp's 32 tensor-memory lanes (the
// 16-token tile's share of one phase).
__device__ __forceinline__ void tc_ld4(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
template <int CW>
__device__ __forceinline__ void tc_ldn(uint32_t taddr, float (&v)[CW]) {
    static_assert(CW == 4 || CW == 32, "tensor-memory load width");
    if constexpr (CW == 4)
        tc_ld4(taddr, v);
    else
        tc_ld32(taddr, v);
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map,
                                            int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::"
        "bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows
// of 128 bytes in 8-row (1024-byte) atoms.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3fffu);  // start address
    d |= (uint64_t)1 << 16;                   // leading byte offset (unused)
    d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows
    d |= (uint64_t)1 << 46;                   // descriptor version
    d |= (uint64_t)2 << 61;                   // swizzle: 128 bytes
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, both K-major,
// N = NT tokens, M = 128 rows.
template <int NT>
__device__ __forceinline__ constexpr uint32_t qmm_idesc() {
    return (1u << 4)                           // D format f32
           | (0u << 7) | (0u << 10)            // A, B: f16
           | ((uint32_t)(NT >> 3) << 17)       // N
           | ((uint32_t)(kQmmRows >> 4) << 24);  // M
}

// 32 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, "
        "%7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, "
        "%21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
        "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
        "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
        "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ bool qmm_wait(uint64_t *bar, uint32_t parity,
                                         unsigned int *status, int *fail) {
    if (mbar_wait_sleep(bar, parity)) return true;
    atomicAdd(&g_qmm_timeouts, 1u);
    atomicOr(status, kStTimeout);
    *fail = 1;
    return false;
}

// ------------------------------------------------------------ pre-pass
// x_ext[m, :] = fp16 activations of token m times 2^e_m (range_scale of the
// largest |x| and |group sum| of the token) in the dequantizers' k order,
// then the bias columns of its scaled group sums X: Xhi of every group, then
// Xlo, then Xhi again (three sections of G columns), then zero padding;
// tscale[m] = 2^-e_m.  u4 order inside each 8-block: 0 4 1 5 2 6 3 7; u8
// inside each 4-block: 0 2 1 3.  A CTA per token, a thread per 8 inputs (one
// 16-byte load; eight lanes make a group, whose sum they form by shuffles):
// a pass for the scale (a block reduction), a pass (the loads hit the
// cache) for the conversion.
constexpr int kPreThreads = 256;

__device__ __forceinline__ void unpack8(const uint4 u, float (&v)[8]) {
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
    v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
    v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}

// Sum of a group of 64 inputs, eight per lane over eight consecutive lanes
// (every lane of the warp takes part; the result is the same on all eight).
__device__ __forceinline__ float group_sum8(const float (&v)[8]) {
    float X = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    X += __shfl_xor_sync(0xffffffffu, X, 1);
    X += __shfl_xor_sync(0xffffffffu, X, 2);
    X += __shfl_xor_sync(0xffffffffu, X, 4);
    return X;
}

template <int BITS>
__global__ void __launch_bounds__(kPreThreads)
    qmm_prepass_kernel(const uint16_t *__restrict__ x, int64_t M, int K,
                       int64_t kext, __half *xe, float *tscale) {
    __shared__ float s_t[kPreThreads / 32];
    // the projection kernel may start its prologue (it reads weights only
    // until it waits for this grid)
    pdl_launch_dependents();
    const int G = K / 64, C = K / 8;  // groups, 8-input chunks
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + m * K);
        float t = 0.f;
        for (int c0 = 0; c0 < C; c0 += kPreThreads) {
            const int c = c0 + tid;
            float v[8];
            unpack8(c < C ? xr[c] : make_uint4(0u, 0u, 0u, 0u), v);
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
            t = fmaxf(t, fmaxf(mx, fabsf(group_sum8(v))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
        if (lane == 0) s_t[warp] = t;
        __syncthreads();
        t = s_t[0];
#pragma unroll
        for (int w = 1; w < kPreThreads / 32; ++w) t = fmaxf(t, s_t[w]);
        __syncthreads();  // s_t is reused by the next token
        float up, down;
        range_scale(t, up, down);
        if (tid == 0) tscale[m] = down;
        __half *row = xe + m * kext;
        for (int c0 = 0; c0 < C; c0 += kPreThreads) {
            const int c = c0 + tid;
            float v[8];
            unpack8(c < C ? xr[c] : make_uint4(0u, 0u, 0u, 0u), v);
            const float X = group_sum8(v);
            if (c >= C) continue;
            uint32_t o[4];
            if constexpr (BITS == 4) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o[i] = h2_bits(__floats2half2_rn(v[i] * up, v[i + 4] * up));
            } else {
                o[0] = h2_bits(__floats2half2_rn(v[0] * up, v[2] * up));
                o[1] = h2_bits(__floats2half2_rn(v[1] * up, v[3] * up));
                o[2] = h2_bits(__floats2half2_rn(v[4] * up, v[6] * up));
                o[3] = h2_bits(__floats2half2_rn(v[5] * up, v[7] * up));
            }
            reinterpret_cast<uint4 *>(row)[c] = make_uint4(o[0], o[1], o[2], o[3]);
            if ((c & 7) == 0) {
                const int g = c >> 3;
                const float Xs = X * up;
                const __half xh = __float2half_rn(Xs);
                const __half xl = __float2half_rn(Xs - __half2float(xh));
                row[K + g] = xh;
                row[K + G + g] = xl;
                row[K + 2 * G + g] = xh;
            }
        }
        for (int64_t c = K + 3 * G + tid; c < kext; c += kPreThreads)
            row[c] = __float2half_rn(0.f);
    }
}

// ------------------------------------------------------------ main kernel
struct QmmParams {
    int64_t M;
    int K;
    int nkb;             // K blocks including the bias blocks
    int G;
    const uint16_t *sc;  // [N, G] (bias blocks read it directly)
    const uint16_t *bi;
    int64_t N;           // weight rows
    int64_t I;           // gate+up: N / 2
    int mode;            // 0 plain, 1 sections, 2 gate+up, 3 sections + RoPE
    uint16_t *y;
    int nsec;
    int64_t sec_start[kMaxSections + 1];
    uint16_t *sec_out[kMaxSections];
    const uint16_t *sec_bias[kMaxSections];
    int rope_hd;
    int64_t rope_end;
    const float2 *rope_cs;
    const float *tscale;  // [M]: 2^-e_m of each token (pre-pass)
    unsigned int *status;
    int ks;               // CTAs per cluster splitting a tile's K blocks
};

// Shared-memory layout (1024-byte aligned regions).
template <int BITS, int NT>
struct QmmLayout {
    static constexpr int AW = BITS == 4 ? 32 : 64;  // A columns per K block
    // ring slots: an activation tile and a K block's A columns each; tensor
    // memory holds NT accumulator columns and the A slots, shared memory the
    // tiles (six tiles at 256 tokens, 213 KB per CTA, ran slower than four)
    static constexpr int SA = (512 - NT) / AW;
    static constexpr int SX = NT == 256 ? 4 : 8;
    static constexpr int KP = NT <= 16 ? 2 : 1;          // K blocks per slot
    static constexpr int RS = (SA < SX ? SA : SX) / KP * KP;  // K blocks
    static constexpr int RP = RS / KP;                   // slots
    // code tiles; a smaller footprint leaves more of the SM's 256 KB to L1
    // (the rows' range scan and the bias blocks read scales and biases
    // through it), and above ~180 KB per CTA the kernel ran slower
    static constexpr int WS = 4;
    static constexpr int XBYTES = NT * 128;           // 64 fp16 per token
    static constexpr int WBYTES = kQmmRows * BITS * 8;  // 64 codes per row
    static constexpr int SBYTES = kQmmRows * 16;      // 8 bf16 per row
    static constexpr size_t XOFF = 0;
    static constexpr size_t WOFF = XOFF + (size_t)RS * XBYTES;
    static constexpr size_t SOFF = WOFF + (size_t)WS * WBYTES;
    static constexpr size_t BYTES = SOFF + (size_t)kQmmSStages * SBYTES;
    static constexpr size_t SMEM = BYTES + 1024;      // alignment slack
};

// fp16 columns of one code K block for one weight row, in the pre-pass's
// k order.  u4: 8 words -> 32 columns; u8: 16 words -> 32 columns of
// 16s(qh-8) and 32 of s(ql-8).
template <int BITS>
__device__ __forceinline__ void dequant_row(const uint32_t *w, float s,
                                            uint32_t *hi, uint32_t *lo) {
    const __half2 off = __floats2half2_rn(1032.f, 1032.f);
    if constexpr (BITS == 4) {
        const __half2 s2 = __floats2half2_rn(s, s);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // (1024 + q_i, 1024 + q_{i+4}) -> s * (q - 8), exact
                uint32_t t = ((w[j] >> (4 * i)) & 0x000f000fu) | 0x64006400u;
                __half2 h = *reinterpret_cast<__half2 *>(&t);
                hi[4 * j + i] = h2_bits(__hmul2(__hsub2(h, off), s2));
            }
    } else {
        const __half2 s1 = __floats2half2_rn(s, s);
        const __half2 s16 = __floats2half2_rn(16.f * s, 16.f * s);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            // bytes (q0, q1, q2, q3); pairs in k order (0,2) (1,3)
            uint32_t l0 = (w[j] & 0x000f000fu) | 0x64006400u;
            uint32_t l1 = ((w[j] >> 8) & 0x000f000fu) | 0x64006400u;
            uint32_t h0 = ((w[j] >> 4) & 0x000f000fu) | 0x64006400u;
            uint32_t h1 = ((w[j] >> 12) & 0x000f000fu) | 0x64006400u;
            hi[2 * j] = h2_bits(
                __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&h0), off), s16));
            hi[2 * j + 1] = h2_bits(
                __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&h1), off), s16));
            lo[2 * j] = h2_bits(
                __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&l0), off), s1));
            lo[2 * j + 1] = h2_bits(
                __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&l1), off), s1));
        }
    }
}

// Bias block (K block kb >= G) for row n: column pair c holds bias columns
// 2c, 2c+1 of the block; bias column j is group j mod G of section j / G,
// which holds the hi part of 2^f_n b' (sections 0 and 1) or its lo part
// (section 2), b' = b + 8s or b + 136s, up = 2^f_n.  G is a multiple of 8,
// so each run of 8 columns is 8 consecutive groups of one section.
template <int BITS>
__device__ __forceinline__ void bias_row(const QmmParams &p, int64_t n, int kb,
                                         float up, uint32_t *a) {
    const int base = (kb - p.G) * 64;
    const float k8 = BITS == 4 ? 8.f : 136.f;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        const int j0 = base + 8 * c8;
        const int t = j0 / p.G, g0 = j0 - t * p.G;
        float e[8];
        if (n >= 0 && t < 3) {
            const uint4 sv = *reinterpret_cast<const uint4 *>(p.sc + n * p.G + g0);
            const uint4 bv = *reinterpret_cast<const uint4 *>(p.bi + n * p.G + g0);
            const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
            const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t sb = i & 1 ? sw[i >> 1] >> 16 : sw[i >> 1] & 0xffffu;
                const uint32_t bb = i & 1 ? bw[i >> 1] >> 16 : bw[i >> 1] & 0xffffu;
                const float bp = fmaf(k8, bf16_bits_to_f32((uint16_t)sb),
                                      bf16_bits_to_f32((uint16_t)bb)) * up;
                const float hi = __half2float(__float2half_rn(bp));
                e[i] = t < 2 ? hi : bp - hi;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            a[4 * c8 + i] = h2_bits(__floats2half2_rn(e[2 * i], e[2 * i + 1]));
    }
}

// SPLIT: launched in clusters that split each tile's K blocks (p.ks CTAs);
// without it the split's code compiles away.
template <int BITS, int NT, bool SPLIT>
__global__ void __launch_bounds__(kQmmThreads, 1)
    qmm_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                  const __grid_constant__ CUtensorMap wmap,
                  const __grid_constant__ CUtensorMap smap, QmmParams p) {
    using L = QmmLayout<BITS, NT>;
    constexpr int AW = L::AW, RS = L::RS, RP = L::RP, KP = L::KP;
    constexpr int WS = L::WS, SS = kQmmSStages;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    // ready[s]: the slot's activation tiles landed and the dequantizing warps
    // (four per K block) stored its A columns; done[s]: its MMAs completed.
    // K block kb sits in slot (kb / KP) % RP, its tile and A columns at
    // position kb % RS.
    __shared__ uint64_t ready[RP], done[RP], wfull[WS], wempty[WS];
    __shared__ uint64_t sfull[SS], sempty[SS], dfull;
    __shared__ uint32_t s_tmem;
    __shared__ int s_xn, s_wn, s_sn;  // TMA loads issued per ring
    __shared__ int s_fail;            // a wait of this CTA ran out
    __shared__ float s_rowt[4][kQmmRows];  // per phase: part of a row's range
    __shared__ float s_tok[NT];            // the tile's tokens' 2^-e_m

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.y * NT;
    const bool gate_up = p.mode == 2;
    // K split: the ks CTAs of a cluster share a tile, rank j taking K blocks
    // [kb0, kb1) (whole runs of 8, so a scale tile never straddles two
    // CTAs); rank 0 adds the others' partial sums and writes the outputs
    const int ks = SPLIT ? p.ks : 1;
    const int rank = SPLIT ? (int)cluster_rank() : 0;
    const int tile = SPLIT ? (int)blockIdx.x / ks : (int)blockIdx.x;
    int kb0 = 0, kb1 = p.nkb;
    if (SPLIT) {
        const int n8 = (p.nkb + 7) / 8;
        kb0 = min(p.nkb, rank * n8 / ks * 8);
        kb1 = min(p.nkb, (rank + 1) * n8 / ks * 8);
    }
    const int nb = kb1 - kb0;  // this CTA's K blocks (an even count)
    // first row of the tile (gate+up: first gate/up pair)
    const int64_t r0 = (int64_t)tile * (gate_up ? kQmmRows / 2 : kQmmRows);
    const int G = p.G;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RP; ++i) {
            mbar_init(&ready[i], 1 + KP * 4);
            mbar_init(&done[i], 1);
        }
        for (int i = 0; i < WS; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], 4);
        }
        for (int i = 0; i < SS; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], kQmmDeqWarps);
        }
        mbar_init(&dfull, 1);
        fence_mbar_init();
        s_xn = s_wn = s_sn = s_fail = 0;
        const CUtensorMap *maps[3] = {&xmap, &wmap, &smap};
        for (int i = 0; i < 3; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(
                             reinterpret_cast<uint64_t>(maps[i]))
                         : "memory");
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t tmem_d = tmem;       // accumulators: cols [0, NT)
    const uint32_t tmem_a = tmem + NT;  // A stages

    // a dequantizing thread's row (the other warps do not use these)
    const int q = warp & 3;                // tensor-memory lane quarter
    const int ph = (warp - kQmmDeq0) / 4;  // local K blocks ph, ph+4, ...
    const int r = q * 32 + lane;           // row within the tile
    int64_t n;                             // weight row (-1: none)
    if (gate_up) {
        const int64_t i = r0 + (r & 63);
        n = i < p.I ? (r < 64 ? i : p.I + i) : -1;
    } else {
        n = r0 + r < p.N ? r0 + r : -1;
    }
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    float rup = 1.f, rdown = 1.f;  // 2^f_n, 2^-f_n
    bool fin = false;              // the accumulators are complete

    if (warp == 0) {
        // -------------------------------------------- activation loader
        if (lane == 0) {
            pdl_wait_primary();  // the tiles are the pre-pass's output
            for (int kp = 0; kp < nb / KP; ++kp) {
                const int s = kp % RP;
                if (kp >= RP &&
                    !qmm_wait(&done[s], ((kp / RP) & 1) ^ 1, p.status, &s_fail))
                    break;
                mbar_expect_tx(&ready[s], KP * L::XBYTES);
                for (int h = 0; h < KP; ++h) {
                    const int lb = KP * kp + h;  // local K block
                    tma_load_2d(smem + L::XOFF + (size_t)(lb % RS) * L::XBYTES,
                                &xmap, (kb0 + lb) * 64, (int)m0, &ready[s]);
                }
                s_xn = KP * kp + KP;
            }
        }
    } else if (warp == 2) {
        // -------------------------------------------- code and scale loader
        if (lane == 0) {
            const int rows = gate_up ? kQmmRows / 2 : kQmmRows;
            for (int kb = kb0; kb < min(kb1, G); ++kb) {
                const int lb = kb - kb0;  // local K block
                if (kb % 8 == 0) {
                    // scale tiles of K blocks kb .. kb+7 (the code blocks'
                    // biases enter through the bias columns)
                    const int sb = lb / 8, s = sb % SS;
                    if (sb >= SS &&
                        !qmm_wait(&sempty[s], ((sb / SS) & 1) ^ 1, p.status, &s_fail))
                        break;
                    unsigned char *ds = smem + L::SOFF + (size_t)s * L::SBYTES;
                    mbar_expect_tx(&sfull[s], L::SBYTES);
                    tma_load_2d(ds, &smap, kb, (int)r0, &sfull[s]);
                    if (gate_up)
                        tma_load_2d(ds + rows * 16, &smap, kb, (int)(p.I + r0),
                                    &sfull[s]);
                    s_sn = sb + 1;
                }
                // packed codes of the tile's rows
                const int s = lb % WS;
                if (lb >= WS &&
                    !qmm_wait(&wempty[s], ((lb / WS) & 1) ^ 1, p.status, &s_fail))
                    break;
                unsigned char *dw = smem + L::WOFF + (size_t)s * L::WBYTES;
                const int wx = kb * BITS * 2;  // 32-bit words
                mbar_expect_tx(&wfull[s], L::WBYTES);
                tma_load_2d(dw, &wmap, wx, (int)r0, &wfull[s]);
                if (gate_up)
                    tma_load_2d(dw + rows * BITS * 8, &wmap, wx, (int)(p.I + r0),
                                &wfull[s]);
                s_wn = lb + 1;
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = qmm_idesc<NT>();
            // descriptor of slot 0's tile; a slot, and 16 columns within
            // it, move the start address (in 16-byte units) only
            const uint64_t desc0 = smem_desc_sw128(smem_u32(smem + L::XOFF));
            // unrolled over the ring's slots, so that a slot's barriers,
            // tiles and A columns are constants (the lone issuing thread's
            // instructions are the loop's cost)
            const int nkp = nb / KP;
            bool ok = true;
            for (int base = 0; ok && base < nkp; base += RP) {
                const uint32_t par = (base / RP) & 1;
#pragma unroll
                for (int s = 0; s < RP; ++s) {
                    const int kp = base + s;
                    if (kp >= nkp) break;
                    if (!qmm_wait(&ready[s], par, p.status, &s_fail)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < KP; ++h) {
                        // local K block lb, at position t = lb % RS
                        const int lb = KP * kp + h, kb = kb0 + lb, t = KP * s + h;
                        const uint64_t bd = desc0 + (uint64_t)(t * (L::XBYTES >> 4));
                        const uint32_t a = tmem_a + t * AW;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_ts(tmem_d, a + kk * 8, bd + 2 * kk, idesc, lb | kk);
                        if (BITS == 8 && kb < G)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc_mma_ts(tmem_d, a + 32 + kk * 8, bd + 2 * kk, idesc, 1u);
                    }
                    tc_commit(&done[s]);
                }
            }
            // always signal the epilogue once every issued MMA is done
            tc_commit(&dfull);
        }
    } else {
        // -------------------------------------------- dequantizers
        // The row's range (see the file comment): the largest |s| * 8 (u4)
        // or 128 (u8) and |b'| over its groups, the four phases' threads of
        // a row taking every fourth 8-group piece of its scales and biases.
        {
            const float qf = BITS == 4 ? 8.f : 128.f;
            const float k8 = BITS == 4 ? 8.f : 136.f;
            float t = 0.f;
            if (n >= 0)
                for (int c = ph; c < G / 8; c += 4) {
                    const uint4 sv = reinterpret_cast<const uint4 *>(p.sc + n * G)[c];
                    const uint4 bv = reinterpret_cast<const uint4 *>(p.bi + n * G)[c];
                    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
                    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float s0 = bf16_lo(sw[i]), s1 = bf16_hi(sw[i]);
                        const float b0 = bf16_lo(bw[i]), b1 = bf16_hi(bw[i]);
                        t = fmaxf(t, fmaxf(fabsf(s0) * qf, fabsf(s1) * qf));
                        t = fmaxf(t, fmaxf(fabsf(fmaf(k8, s0, b0)),
                                           fabsf(fmaf(k8, s1, b1))));
                    }
                }
            s_rowt[ph][r] = t;
        }
        asm volatile("bar.sync 2, %0;" ::"r"(kQmmDeqWarps * kWarp) : "memory");
        range_scale(fmaxf(fmaxf(s_rowt[0][r], s_rowt[1][r]),
                          fmaxf(s_rowt[2][r], s_rowt[3][r])),
                    rup, rdown);
        // The block's A columns into its ring slot, once its previous MMAs
        // are done (false: a wait ran out).
        auto store_a = [&](int lb, const uint32_t (&hi)[32],
                           const uint32_t (&lo)[BITS == 8 ? 32 : 1]) {
            const int sa = lb % RS, kp = lb / KP, sp = kp % RP;
            // warp-uniform: tcgen05.st below is a warp-collective
            if (kp >= RP &&
                !__all_sync(0xffffffffu, qmm_wait(&done[sp], ((kp / RP) & 1) ^ 1,
                                                  p.status, &s_fail)))
                return false;
            const uint32_t col = tmem_a + sa * AW + lane_off;
            tc_st32(col, hi);
            if constexpr (BITS == 8) tc_st32(col + 32, lo);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ready[sp]);
            return true;
        };
        // code blocks, then bias blocks (two loops keep the bias columns'
        // code out of the hot loop); local K blocks ph, ph + 4, ...
        int lb = ph;
        bool ok = true;
        for (; ok && lb < nb && kb0 + lb < G; lb += 4) {
            const int kb = kb0 + lb;
            uint32_t hi[32], lo[BITS == 8 ? 32 : 1];
            const int ss = (lb / 8) % SS;
            if ((kb & 7) == ph &&
                !__all_sync(0xffffffffu, qmm_wait(&sfull[ss], (lb / 8 / SS) & 1,
                                                  p.status, &s_fail))) {
                ok = false;
                break;
            }
            const int sw = lb % WS;
            if (!__all_sync(0xffffffffu,
                            qmm_wait(&wfull[sw], (lb / WS) & 1, p.status, &s_fail))) {
                ok = false;
                break;
            }
            const uint4 *ws = reinterpret_cast<const uint4 *>(
                smem + L::WOFF + (size_t)sw * L::WBYTES + (size_t)r * BITS * 8);
            uint32_t w[BITS * 2];
            if constexpr (BITS == 4) {
                // rows 128 bytes apart read their two 16-byte chunks in
                // opposite order (different banks in one instruction)
                const bool rot = (r >> 2) & 1;
                const uint4 c0 = ws[rot ? 1 : 0], c1 = ws[rot ? 0 : 1];
                const uint4 lo4 = rot ? c1 : c0, hi4 = rot ? c0 : c1;
                w[0] = lo4.x; w[1] = lo4.y; w[2] = lo4.z; w[3] = lo4.w;
                w[4] = hi4.x; w[5] = hi4.y; w[6] = hi4.z; w[7] = hi4.w;
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 c = ws[v];
                    w[4 * v] = c.x; w[4 * v + 1] = c.y;
                    w[4 * v + 2] = c.z; w[4 * v + 3] = c.w;
                }
            }
            const uint16_t *st = reinterpret_cast<const uint16_t *>(
                smem + L::SOFF + (size_t)ss * L::SBYTES);
            const float s = bf16_bits_to_f32(st[r * 8 + (kb & 7)]) * rup;
            // the codes and scale of this block are in registers
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&wempty[sw]);
                if ((kb & 7) == 4 + ph || kb == G - 1) mbar_arrive(&sempty[ss]);
            }
            dequant_row<BITS>(w, s, hi, lo);
            ok = store_a(lb, hi, lo);
        }
        for (; ok && lb < nb; lb += 4) {
            uint32_t hi[32], lo[BITS == 8 ? 32 : 1];
            bias_row<BITS>(p, n, kb0 + lb, rup, hi);
            if constexpr (BITS == 8)
#pragma unroll
                for (int i = 0; i < 32; ++i) lo[i] = 0u;
            ok = store_a(lb, hi, lo);
        }
        // all MMAs done
        fin = __all_sync(0xffffffffu, qmm_wait(&dfull, 0, p.status, &s_fail));
        if (fin) tc_fence_after();
        {
            // the tile's token factors, the pre-pass's output
            pdl_wait_primary();
            const int tix = threadIdx.x - kQmmDeq0 * kWarp;
            for (int i = tix; i < NT; i += kQmmDeqWarps * kWarp)
                s_tok[i] = m0 + i < p.M ? p.tscale[m0 + i] : 0.f;
            asm volatile("bar.sync 2, %0;" ::"r"(kQmmDeqWarps * kWarp) : "memory");
        }
        if (SPLIT && rank > 0 && fin) {
            // this CTA's partial sums, for rank 0 to add: red[c][r] (fp32)
            float *red = reinterpret_cast<float *>(smem + L::XOFF);
            static_assert((size_t)NT * kQmmRows * 4 <= (size_t)L::RS * L::XBYTES,
                          "the partial sums must fit in the activation ring");
            constexpr int CW = NT / 4 < 32 ? NT / 4 : 32;
            for (int c0 = ph * (NT / 4); c0 < (ph + 1) * (NT / 4); c0 += CW) {
                float d[CW];
                tc_ldn<CW>(tmem_d + lane_off + c0, d);
#pragma unroll
                for (int j = 0; j < CW; ++j) red[(c0 + j) * kQmmRows + r] = d[j];
            }
        }
    }
    // every thread of the cluster: the partial sums are in place
    if (SPLIT) cluster_sync_all();
    if (warp >= kQmmDeq0 && rank == 0) {
        // -------------------------------------------- epilogue
        // accumulators are 2^(f_n + e_m) times the outputs: d * 2^-f_n * 2^-e_m
        const int c_lo = ph * (NT / 4), c_hi = c_lo + NT / 4;
        // columns a phase reads at a time: 32, or its whole share of a
        // 16-token tile
        constexpr int CW = NT / 4 < 32 ? NT / 4 : 32;
        // this CTA's accumulators plus, under a K split, the other ranks'
        // partial sums (distributed shared memory)
        auto load_acc = [&](int c0, float (&v)[CW]) {
            tc_ldn<CW>(tmem_d + lane_off + c0, v);
            if (SPLIT) {
                const float *red = reinterpret_cast<const float *>(smem + L::XOFF);
                for (int j2 = 1; j2 < ks; ++j2) {
                    float t[CW];
                    ld_cluster_f32_n<CW>(red + c0 * kQmmRows + r, (uint32_t)j2,
                                         kQmmRows, t);
#pragma unroll
                    for (int j = 0; j < CW; ++j) v[j] += t[j];
                }
            }
        };
        if (gate_up) {
            // gate warps (rows 0-63) hand their accumulators to the up
            // warps through the (now idle) activation ring
            float *gbuf = reinterpret_cast<float *>(smem + L::XOFF);
            constexpr int GS = NT + 1;  // padded row stride: no bank conflicts
            if (fin && r < 64) {
                for (int c0 = c_lo; c0 < c_hi; c0 += CW) {
                    float g[CW];
                    load_acc(c0, g);
#pragma unroll
                    for (int j = 0; j < CW; ++j)
                        gbuf[r * GS + c0 + j] = g[j] * rdown * s_tok[c0 + j];
                }
            }
            asm volatile("bar.sync 2, %0;" ::"r"(kQmmDeqWarps * kWarp) : "memory");
            if (fin && r >= 64) {
                const int pr = r - 64;
                const int64_t i = r0 + pr;
                for (int c0 = c_lo; c0 < c_hi; c0 += CW) {
                    float u[CW];
                    load_acc(c0, u);
                    if (i >= p.I) continue;
                    for (int j = 0; j < CW; ++j) {
                        const int64_t m = m0 + c0 + j;
                        if (m >= p.M) break;
                        const float g = gbuf[pr * GS + c0 + j];
                        const float uv = u[j] * rdown * s_tok[c0 + j];
                        p.y[m * p.I + i] =
                            // SiLU with the fast divide (two ulps; the
                            // output is bf16; 0 once e^-g passes 2^126)
                            f32_to_bf16_bits(__fdividef(g, 1.0f + __expf(-g)) * uv);
                    }
                }
            }
        } else if (p.mode == 3) {
            // rotary embedding: a row and its partner (i, i + d/2 of one
            // head, in this tile as d divides 128) exchange their values
            // through the (now idle) rings, padded rows of NT + 1 floats
            float *buf = reinterpret_cast<float *>(smem + L::XOFF);
            constexpr int GS = NT + 1;
            static_assert((size_t)kQmmRows * GS * 4 <= L::BYTES,
                          "the exchange rows must fit in the rings");
            int sidx = 0;
            float bias = 0.f;
            if (n >= 0) {
                while (sidx + 1 < p.nsec && n >= p.sec_start[sidx + 1]) ++sidx;
                if (p.sec_bias[sidx])
                    bias = bf16_bits_to_f32(
                        p.sec_bias[sidx][n - p.sec_start[sidx]]);
            }
            if (fin) {
                for (int c0 = c_lo; c0 < c_hi; c0 += CW) {
                    float d[CW];
                    load_acc(c0, d);
#pragma unroll
                    for (int j = 0; j < CW; ++j)
                        buf[r * GS + c0 + j] = d[j] * rdown * s_tok[c0 + j] + bias;
                }
            }
            asm volatile("bar.sync 2, %0;" ::"r"(kQmmDeqWarps * kWarp) : "memory");
            if (fin && n >= 0) {
                const int half = p.rope_hd / 2;
                const int rr = r % p.rope_hd;
                const bool first = rr < half;
                const int pr = first ? r + half : r - half;
                const int i = first ? rr : rr - half;
                const bool rot = n < p.rope_end;
                const int64_t jj = n - p.sec_start[sidx];
                const int64_t size = p.sec_start[sidx + 1] - p.sec_start[sidx];
                constexpr int RW = NT / 4 < 16 ? NT / 4 : 16;
                for (int c0 = c_lo; c0 < c_hi; c0 += RW) {
                    // RW (cos, sin) loads in flight together
                    float2 tv[RW];
#pragma unroll
                    for (int j = 0; j < RW; ++j) {
                        const int64_t m = min(m0 + c0 + j, p.M - 1);
                        tv[j] = rot ? p.rope_cs[m * half + i]
                                    : make_float2(1.0f, 0.0f);
                    }
#pragma unroll
                    for (int j = 0; j < RW; ++j) {
                        const int64_t m = m0 + c0 + j;
                        if (m < p.M) {
                            const float own = buf[r * GS + c0 + j];
                            const float oth = buf[pr * GS + c0 + j];
                            const float val = first ? own * tv[j].x - oth * tv[j].y
                                                    : own * tv[j].x + oth * tv[j].y;
                            p.sec_out[sidx][m * size + jj] = f32_to_bf16_bits(val);
                        }
                    }
                }
            }
        } else if (fin) {
            int sidx = 0;
            if (p.mode == 1 && n >= 0)
                while (sidx + 1 < p.nsec && n >= p.sec_start[sidx + 1]) ++sidx;
            for (int c0 = c_lo; c0 < c_hi; c0 += CW) {
                float d[CW];
                load_acc(c0, d);
                if (n < 0) continue;
                for (int j = 0; j < CW; ++j) {
                    const int64_t m = m0 + c0 + j;
                    if (m >= p.M) break;
                    const float dv = d[j] * rdown * s_tok[c0 + j];
                    if (p.mode == 0) {
                        p.y[m * p.N + n] = f32_to_bf16_bits(dv);
                    } else {
                        const int64_t jj = n - p.sec_start[sidx];
                        const int64_t size =
                            p.sec_start[sidx + 1] - p.sec_start[sidx];
                        float val = dv;
                        if (p.sec_bias[sidx])
                            val += bf16_bits_to_f32(p.sec_bias[sidx][jj]);
                        p.sec_out[sidx][m * size + jj] = f32_to_bf16_bits(val);
                    }
                }
            }
        }
    }
    // the other ranks keep their shared memory until rank 0 has read it
    if (SPLIT) cluster_sync_all();

    // ------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && s_fail) {
        // nothing may still be landing in shared memory or tensor memory.
        // Unless a wait ran out, every load was waited for by its consumer
        // and the last MMA completed (dfull), so there is nothing to check;
        // otherwise wait for the last loads of each ring.
        // A slot's ready phase also needs its dequantizers' arrivals, so
        // after a wait that ran out it may never complete; but the
        // activation loader issues a tile only once the slot's previous
        // MMAs are done, so every tile it issued either was consumed or
        // preceded one of its own waits running out (2 s): by now it has
        // landed, and a short bounded wait suffices
        for (int k = max(0, s_xn - RS); k < s_xn; k += KP)
            if (!mbar_wait(&ready[(k / KP) % RP], ((k / KP) / RP) & 1, 1000000ull))
                break;
        for (int k = max(0, s_wn - WS); k < s_wn; ++k)
            if (!mbar_wait(&wfull[k % WS], (k / WS) & 1)) break;
        for (int k = max(0, s_sn - SS); k < s_sn; ++k)
            if (!mbar_wait(&sfull[k % SS], (k / SS) & 1)) break;
        mbar_wait(&dfull, 0);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr,
                                             12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D tensor map over a row-major [rows, cols] array.
static int encode_2d(CUtensorMap *map, CUtensorMapDataType type, int esize,
                     const void *base, int64_t cols, int64_t rows,
                     uint32_t box_cols, uint32_t box_rows,
                     CUtensorMapSwizzle swz, const char *what) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode)
        return set_error(GWA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)cols * esize};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    CUresult cr = encode(map, type, 2, const_cast<void *>(base), gdim, gstride,
                         box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS)
        return set_error(GWA_ERR_CUDA, "tensor map (%s) encode failed (%d)",
                         what, (int)cr);
    return GWA_OK;
}


template <int BITS, int NT>
static int qmm_launch(const QmmArgs &a, unsigned char *ws, cudaStream_t st) {
    using L = QmmLayout<BITS, NT>;
    const int64_t M = a.M, K = a.w.K, G = K / 64;
    const int64_t kext = qmm_kext(K);
    unsigned int *status = reinterpret_cast<unsigned int *>(ws);
    __half *xe = reinterpret_cast<__half *>(ws + kStatusBytes);
    float *tscale = reinterpret_cast<float *>(ws + kStatusBytes + qmm_xe_bytes(M, K));

    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm status reset: %s",
                         cudaGetErrorString(e));
    // a CTA per token (a thread per 8 inputs)
    int64_t pblocks = M;
    if (pblocks > (int64_t)num_sms() * 8) pblocks = (int64_t)num_sms() * 8;
    qmm_prepass_kernel<BITS><<<(unsigned)pblocks, kPreThreads, 0, st>>>(
        a.x, M, (int)K, kext, xe, tscale);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm pre-pass: %s", cudaGetErrorString(e));

    const bool gate_up = a.mode == 2;
    const uint32_t box_rows = gate_up ? kQmmRows / 2 : kQmmRows;
    CUtensorMap xmap, wmap, smap;
    int rc = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xe, kext, M,
                       64, NT, CU_TENSOR_MAP_SWIZZLE_128B, "activations");
    if (!rc)
        rc = encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, a.w.wq,
                       K * BITS / 32, a.w.N, BITS * 2, box_rows,
                       CU_TENSOR_MAP_SWIZZLE_NONE, "codes");
    if (!rc)
        rc = encode_2d(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, a.w.scales, G,
                       a.w.N, 8, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE,
                       "scales");
    if (rc) return rc;

    QmmParams p{};
    p.M = M;
    p.K = (int)K;
    p.nkb = (int)(kext / 64);
    p.G = (int)G;
    p.sc = a.w.scales;
    p.bi = a.w.biases;
    p.N = a.w.N;
    p.I = a.w.N / 2;
    p.mode = a.mode;
    p.y = a.y;
    p.nsec = a.nsec;
    const bool secs = a.mode == 1 || a.mode == 3;
    for (int s = 0; s <= a.nsec && secs; ++s) p.sec_start[s] = a.sec_start[s];
    for (int s = 0; s < a.nsec && secs; ++s) {
        p.sec_out[s] = a.sec_out[s];
        p.sec_bias[s] = a.sec_bias[s];
    }
    p.rope_hd = a.rope_hd;
    p.rope_end = a.rope_end;
    p.rope_cs = a.rope_cs;
    p.tscale = tscale;
    p.status = status;

    auto kern = qmm_tc_kernel<BITS, NT, false>;
    auto kern_split = qmm_tc_kernel<BITS, NT, true>;
    int resident = 0;
    e = occupancy_grid(reinterpret_cast<const void *>(kern), kQmmThreads,
                       L::SMEM, &resident);
    if (e == cudaSuccess)
        e = occupancy_grid(reinterpret_cast<const void *>(kern_split), kQmmThreads,
                           L::SMEM, &resident);
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm setup: %s", cudaGetErrorString(e));
    const int64_t rows = gate_up ? p.I : p.N;
    const int64_t row_tiles = (rows + box_rows - 1) / box_rows;
    const int64_t tiles = row_tiles * ((M + NT - 1) / NT);
    // K split over a cluster of ks CTAs when the tiles leave SMs idle: the
    // largest ks whose clusters all fit in one wave, each CTA taking 1/ks of
    // a tile's K blocks.  (Splits that need a second wave of clusters lost:
    // each CTA also pays the prologue, the partial sums' exchange and, on
    // rank 0, the epilogue; at 512 tokens a 3-way split of 80 tiles took
    // o_proj from 40 to 57 us.)
    p.ks = 1;
    if (tiles < resident) {
        const int n8 = (p.nkb + 7) / 8;
        for (int ks = 2; ks <= kQmmMaxSplit && n8 >= 2 * ks; ++ks) {
            const int cap = resident_clusters(
                reinterpret_cast<const void *>(kern_split), ks, kQmmThreads, L::SMEM);
            if (cap >= tiles) p.ks = ks;
        }
    }
    dim3 grid((unsigned)(row_tiles * p.ks), (unsigned)((M + NT - 1) / NT));
    // programmatic dependent launch: the prologue (barriers, tensor memory,
    // the rows' ranges from the scales) and the first code tiles overlap
    // the pre-pass; the kernel waits for it before touching its output
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kQmmThreads);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = p.ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.ks > 1 ? 2 : 1;
    e = p.ks > 1 ? cudaLaunchKernelEx(&cfg, kern_split, xmap, wmap, smap, p)
                 : cudaLaunchKernelEx(&cfg, kern, xmap, wmap, smap, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm launch: %s", cudaGetErrorString(e));
    return GWA_OK;
}

bool qmm_eligible(const QmmArgs &a) {
    auto a16 = [](const void *q) {
        return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
    };
    // the scale tiles need rows of whole 16-byte units (K/64 a multiple of
    // 8); TMA wants 16-byte aligned bases
    return a.w.group == 64 && (a.w.K / 64) % 8 == 0 && a16(a.w.wq) &&
           a16(a.w.scales) &&
           a16(a.w.biases) && a.M <= 0x7fffffffLL && a.w.N <= 0x7fffffffLL &&
           (a.w.bits == 4 || a.w.bits == 8);
}

int qmm_run(const QmmArgs &a, void *workspace, size_t workspace_bytes,
            cudaStream_t st) {
    const size_t need = qmm_workspace_bytes(a.M, a.w.K);
    if (!workspace || workspace_bytes < need)
        return set_error(GWA_ERR_WORKSPACE,
                         "M=%lld K=%lld needs %zu bytes of workspace (got %zu)",
                         (long long)a.M, (long long)a.w.K, need,
                         workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return set_error(GWA_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    if (a.M > 0x7fffffffLL)
        return set_error(GWA_ERR_INVALID_ARG, "M too large");
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    // 256-token tiles once there are enough; 16-token tiles for up to 16
    // tokens (an MMA of N = 16: the tensor pipe does 8 times less padding
    // work than at 128)
    if (a.M <= 16)
        return a.w.bits == 4 ? qmm_launch<4, 16>(a, ws, st)
                             : qmm_launch<8, 16>(a, ws, st);
    const bool wide = a.M > 128;
    if (a.w.bits == 4)
        return wide ? qmm_launch<4, 256>(a, ws, st) : qmm_launch<4, 128>(a, ws, st);
    return wide ? qmm_launch<8, 256>(a, ws, st) : qmm_launch<8, 128>(a, ws, st);
}

unsigned int qmm_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_qmm_timeouts, sizeof v);
    if (reset) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_qmm_timeouts, &z, sizeof z);
    }
    return v;
}

}  // namespace gwa
