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
// three extra columns per group (b'hi*Xhi + b'hi*Xlo + b'lo*Xhi).  Activations
// are converted to fp16 once per call by a pre-pass (exact for |x| in fp16's
// normal range); products are exact and accumulate in fp32 in tensor memory.
//
// Kernel shape.  A CTA computes two 128-row weight tiles (for gate+up: the
// gate tile and the matching up tile) against 128 tokens:
//   warp 0    allocates tensor memory, loads the activation tile of each
//             64-wide K block with TMA (128-byte swizzle) into a smem ring;
//   warp 1    issues tcgen05.mma (A from tensor memory, B from smem);
//   warps 2-9 dequantize: thread (tile, row) turns its row's 64 codes of the
//             K block into 32 fp16 pairs and writes them to tensor memory
//             with tcgen05.st (the A operand), then reads the fp32
//             accumulators back with tcgen05.ld for the epilogue.
// Every wait is bounded (2 s); a wait that runs out flags the workspace
// status word and the kernel unwinds without hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "qmm.h"

namespace gwa {

constexpr int kQmmThreads = 320;     // 10 warps
constexpr int kQmmTok = 128;         // tokens per CTA (MMA N)
constexpr int kQmmRows = 128;        // rows per weight tile (MMA M)
constexpr int kQmmXStages = 6;       // activation ring depth
constexpr int kXStageBytes = kQmmTok * 64 * 2;   // 16 KB, 128-byte swizzle
constexpr size_t kQmmSmem = 120 * 1024;  // > half an SM: one CTA per SM
constexpr int kStatusBytes = 256;
constexpr int kQmmPrefetch = 4;      // code blocks loaded ahead per thread

// status word bits
constexpr unsigned kStTimeout = 1u;
constexpr unsigned kStFp16Range = 2u;

static __device__ unsigned int g_qmm_timeouts;

static int64_t qmm_kext(int64_t K) {
    const int64_t G = K / 64;
    return K + ((3 * G + 63) / 64) * 64;
}

size_t qmm_workspace_bytes(int64_t M, int64_t K) {
    const size_t x = (size_t)M * (size_t)qmm_kext(K) * 2;
    return kStatusBytes + ((x + 255) / 256) * 256;
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
// N = 128 tokens, M = 128 rows.
constexpr uint32_t kIdesc = (1u << 4)                    // D format f32
                            | (0u << 7) | (0u << 10)     // A, B: f16
                            | ((uint32_t)(kQmmTok >> 3) << 17)
                            | ((uint32_t)(kQmmRows >> 4) << 24);

__device__ __forceinline__ uint32_t h2_bits(__half2 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ bool qmm_wait(uint64_t *bar, uint32_t parity,
                                         unsigned int *status) {
    if (mbar_wait(bar, parity)) return true;
    atomicAdd(&g_qmm_timeouts, 1u);
    atomicOr(status, kStTimeout);
    return false;
}

// ------------------------------------------------------------ pre-pass
// x_ext[m, :] = fp16 activations of token m in the dequantizers' k order,
// then per group g three bias columns (Xhi, Xlo, Xhi), then zero padding.
// u4 order inside each 8-block: 0 4 1 5 2 6 3 7; u8 inside each 4-block:
// 0 2 1 3.  One thread per (token, group).
template <int BITS>
__global__ void qmm_prepass_kernel(const uint16_t *__restrict__ x, int64_t M,
                                   int K, int64_t kext, __half *xe,
                                   unsigned int *status) {
    const int G = K / 64;
    const int64_t items = M * G;
    for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
         it < items; it += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = it / G;
        const int g = (int)(it - m * G);
        const uint4 *src = reinterpret_cast<const uint4 *>(x + m * K + g * 64);
        __half *dst = xe + m * kext + g * 64;
        float v[64];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
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
        float X = 0.f;
        bool over = false;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            X += v[i];
            over |= fabsf(v[i]) > 65504.f;
        }
        uint32_t o[32];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const float *vb = v + 8 * b;
            if constexpr (BITS == 4) {
                o[4 * b + 0] = h2_bits(__floats2half2_rn(vb[0], vb[4]));
                o[4 * b + 1] = h2_bits(__floats2half2_rn(vb[1], vb[5]));
                o[4 * b + 2] = h2_bits(__floats2half2_rn(vb[2], vb[6]));
                o[4 * b + 3] = h2_bits(__floats2half2_rn(vb[3], vb[7]));
            } else {
                o[4 * b + 0] = h2_bits(__floats2half2_rn(vb[0], vb[2]));
                o[4 * b + 1] = h2_bits(__floats2half2_rn(vb[1], vb[3]));
                o[4 * b + 2] = h2_bits(__floats2half2_rn(vb[4], vb[6]));
                o[4 * b + 3] = h2_bits(__floats2half2_rn(vb[5], vb[7]));
            }
        }
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            d4[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        const __half xh = __float2half_rn(X);
        const __half xl = __float2half_rn(X - __half2float(xh));
        __half *bc = xe + m * kext + K + 3 * g;
        bc[0] = xh;
        bc[1] = xl;
        bc[2] = xh;
        over |= fabsf(X) > 65504.f;
        if (over) atomicOr(status, kStFp16Range);
        if (g == 0)
            for (int64_t c = K + 3 * G; c < kext; ++c)
                xe[m * kext + c] = __float2half_rn(0.f);
    }
}

// ------------------------------------------------------------ main kernel
struct QmmParams {
    int64_t M;
    int K;
    int64_t kext;
    int nkb;             // K blocks including the bias blocks
    int G;
    const uint32_t *wq;
    const uint16_t *sc;
    const uint16_t *bi;
    int64_t N;           // weight rows
    int64_t I;           // gate+up: N / 2
    int mode;            // 0 plain, 1 sections, 2 gate+up
    uint16_t *y;
    int nsec;
    int64_t sec_start[kMaxSections + 1];
    uint16_t *sec_out[kMaxSections];
    const uint16_t *sec_bias[kMaxSections];
    unsigned int *status;
};

// Raw inputs of one K block for one weight row: the packed words and the
// group's bf16 scale and bias (code blocks only).
template <int BITS>
struct RawBlock {
    uint4 w[BITS == 4 ? 2 : 4];
    uint16_t s, b;
};

template <int BITS>
__device__ __forceinline__ void load_raw(const QmmParams &p, int64_t n, int kb,
                                         RawBlock<BITS> &r) {
    constexpr int NV = BITS == 4 ? 2 : 4;  // 16-byte vectors per 64 codes
    if (n < 0 || kb >= p.G) return;
    const int64_t wpr = (int64_t)p.K * BITS / 32;
    const uint4 *src =
        reinterpret_cast<const uint4 *>(p.wq + n * wpr) + (int64_t)kb * NV;
#pragma unroll
    for (int i = 0; i < NV; ++i) r.w[i] = ld_stream(src + i);
    r.s = ld_u16(p.sc + n * p.G + kb);
    r.b = ld_u16(p.bi + n * p.G + kb);
}

// fp16 dequantized columns of one K block for one weight row (the A tile
// row), in the k order of the pre-pass.  u4: 32 columns; u8: 64 columns
// (16s(qh-8) in the first 32, s(ql-8) in the last 32).
template <int BITS>
__device__ __forceinline__ void dequant_block(const QmmParams &p, int64_t n,
                                              int kb, const RawBlock<BITS> &r,
                                              uint32_t (&a)[64],
                                              unsigned &flags) {
    constexpr int W = BITS == 4 ? 8 : 16;  // words per 64 codes
    constexpr int NC = BITS == 4 ? 32 : 64;
    if (n < 0) {
#pragma unroll
        for (int i = 0; i < NC; ++i) a[i] = 0u;
        return;
    }
    if (kb < p.G) {
        uint32_t w[W];
#pragma unroll
        for (int i = 0; i < W / 4; ++i) {
            w[4 * i] = r.w[i].x;
            w[4 * i + 1] = r.w[i].y;
            w[4 * i + 2] = r.w[i].z;
            w[4 * i + 3] = r.w[i].w;
        }
        const float s = bf16_bits_to_f32(r.s);
        if (!(fabsf(s) <= 511.f) || (s != 0.f && fabsf(s) < 6.103515625e-05f))
            flags |= kStFp16Range;
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
                    a[4 * j + i] = h2_bits(__hmul2(__hsub2(h, off), s2));
                }
        } else {
            const __half2 s1 = __floats2half2_rn(s, s);
            const __half2 s16 = __floats2half2_rn(16.f * s, 16.f * s);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                // bytes (q0, q1, q2, q3); pairs in k order (0,2) (1,3)
                uint32_t l0 = (w[j] & 0x000f000fu) | 0x64006400u;          // ql0 ql2
                uint32_t l1 = ((w[j] >> 8) & 0x000f000fu) | 0x64006400u;   // ql1 ql3
                uint32_t h0 = ((w[j] >> 4) & 0x000f000fu) | 0x64006400u;   // qh0 qh2
                uint32_t h1 = ((w[j] >> 12) & 0x000f000fu) | 0x64006400u;  // qh1 qh3
                a[2 * j] = h2_bits(
                    __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&h0), off), s16));
                a[2 * j + 1] = h2_bits(
                    __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&h1), off), s16));
                a[32 + 2 * j] = h2_bits(
                    __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&l0), off), s1));
                a[32 + 2 * j + 1] = h2_bits(
                    __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&l1), off), s1));
            }
        }
    } else {
        // bias block: column pair c holds bias columns 2c, 2c+1 of this
        // block; bias column j belongs to group j/3 (hi, hi, lo)
        const int base = (kb - p.G) * 64;
        const float k8 = BITS == 4 ? 8.f : 136.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            float e[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = base + 2 * c + h;
                const int g = j / 3, which = j - 3 * g;
                float val = 0.f;
                if (g < p.G) {
                    const float s = bf16_bits_to_f32(p.sc[n * p.G + g]);
                    const float b = bf16_bits_to_f32(p.bi[n * p.G + g]);
                    const float bp = fmaf(k8, s, b);
                    const float hi = __half2float(__float2half_rn(bp));
                    val = which < 2 ? hi : bp - hi;
                    if (fabsf(bp) > 65504.f) flags |= kStFp16Range;
                }
                e[h] = val;
            }
            a[c] = h2_bits(__floats2half2_rn(e[0], e[1]));
        }
        if constexpr (BITS == 8) {
#pragma unroll
            for (int c = 32; c < 64; ++c) a[c] = 0u;
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kQmmThreads, 1)
    qmm_tc_kernel(const __grid_constant__ CUtensorMap xmap, QmmParams p) {
    constexpr int AW = BITS == 4 ? 32 : 64;     // A columns per tile per block
    constexpr int SA = 256 / (2 * AW);          // A stages in tensor memory
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned ring for the 128-byte swizzle atoms
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t xfull[kQmmXStages], xempty[kQmmXStages];
    __shared__ uint64_t afull[SA], aempty[SA], dfull;
    __shared__ uint32_t s_tmem;
    __shared__ int s_xissued, s_xconsumed;

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.y * kQmmTok;
    const bool gate_up = p.mode == 2;
    const int64_t r0 = (int64_t)blockIdx.x * (gate_up ? kQmmRows : 2 * kQmmRows);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kQmmXStages; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 1);
        }
        for (int i = 0; i < SA; ++i) {
            mbar_init(&afull[i], 8);
            mbar_init(&aempty[i], 1);
        }
        mbar_init(&dfull, 1);
        fence_mbar_init();
        s_xissued = 0;
        s_xconsumed = p.nkb;
        asm volatile("prefetch.tensormap [%0];" ::"l"(
                         reinterpret_cast<uint64_t>(&xmap))
                     : "memory");
    }
    if (warp == 0) tmem_alloc(&s_tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t tmem_d = tmem;          // D0: cols [0,128), D1: [128,256)
    const uint32_t tmem_a = tmem + 256;    // A stages

    if (warp == 0) {
        // -------------------------------------------- activation loader
        if (lane == 0) {
            for (int kb = 0; kb < p.nkb; ++kb) {
                const int s = kb % kQmmXStages;
                if (kb >= kQmmXStages &&
                    !qmm_wait(&xempty[s], ((kb / kQmmXStages) & 1) ^ 1, p.status))
                    break;
                mbar_expect_tx(&xfull[s], kXStageBytes);
                tma_load_2d(smem + s * kXStageBytes, &xmap, kb * 64, (int)m0,
                            &xfull[s]);
                s_xissued = kb + 1;
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------- MMA issuer
        if (lane == 0) {
            int kb = 0;
            for (; kb < p.nkb; ++kb) {
                const int sx = kb % kQmmXStages, sa = kb % SA;
                if (!qmm_wait(&xfull[sx], (kb / kQmmXStages) & 1, p.status) ||
                    !qmm_wait(&afull[sa], (kb / SA) & 1, p.status)) {
                    atomicMin(&s_xconsumed, kb);
                    break;
                }
                tc_fence_after();
                const uint32_t xs = smem_u32(smem + sx * kXStageBytes);
                const int subs = (BITS == 8 && kb < p.G) ? 2 : 1;
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    for (int sub = 0; sub < subs; ++sub)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t a = tmem_a + sa * (2 * AW) + t * AW +
                                               sub * 32 + kk * 8;
                            const uint64_t bdesc = smem_desc_sw128(xs + kk * 32);
                            tc_mma_ts(tmem_d + t * kQmmTok, a, bdesc, kIdesc,
                                      (kb | sub | kk) != 0);
                        }
                tc_commit(&xempty[sx]);
                tc_commit(&aempty[sa]);
            }
            // always signal the epilogue once every issued MMA is done
            tc_commit(&dfull);
        }
    } else {
        // -------------------------------------------- dequantizers
        const int pw = warp - 2;              // 0..7
        const int tile = pw / 4;              // weight tile 0 or 1
        const int q = warp & 3;               // tensor-memory lane quarter
        const int r = q * 32 + lane;          // row within the tile
        int64_t n;                            // weight row
        if (gate_up) {
            const int64_t i = r0 + r;
            n = i < p.I ? (tile ? p.I + i : i) : -1;
        } else {
            const int64_t i = r0 + tile * kQmmRows + r;
            n = i < p.N ? i : -1;
        }
        unsigned flags = 0;
        // A ring of raw code blocks, loaded kQmmPrefetch blocks ahead so
        // the HBM latency of the codes overlaps the tensor-core work.
        RawBlock<BITS> ring[kQmmPrefetch];
#pragma unroll
        for (int i = 0; i < kQmmPrefetch; ++i)
            if (i < p.nkb) load_raw<BITS>(p, n, i, ring[i]);
        bool ok = true;  // pipeline healthy
        for (int kb0 = 0; kb0 < p.nkb && ok; kb0 += kQmmPrefetch) {
#pragma unroll
            for (int i = 0; i < kQmmPrefetch; ++i) {
                const int kb = kb0 + i;
                if (kb >= p.nkb) break;
                const int sa = kb % SA;
                // warp-uniform: tcgen05.st below is a warp-collective
                if (kb >= SA &&
                    !__all_sync(0xffffffffu, qmm_wait(&aempty[sa],
                                                      ((kb / SA) & 1) ^ 1,
                                                      p.status))) {
                    ok = false;
                    break;
                }
                uint32_t a[64];
                dequant_block<BITS>(p, n, kb, ring[i], a, flags);
                if (kb + kQmmPrefetch < p.nkb)
                    load_raw<BITS>(p, n, kb + kQmmPrefetch, ring[i]);
                const uint32_t col = tmem_a + sa * (2 * AW) + tile * AW;
                const uint32_t taddr = col + ((uint32_t)(q * 32) << 16);
                uint32_t v0[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v0[j] = a[j];
                tc_st32(taddr, v0);
                if constexpr (BITS == 8) {
                    uint32_t v1[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v1[j] = a[32 + j];
                    tc_st32(taddr + 32, v1);
                }
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[sa]);
            }
        }
        if (flags) atomicOr(p.status, flags);

        // -------------------------------------------- epilogue
        if (__all_sync(0xffffffffu, qmm_wait(&dfull, 0, p.status))) {
            tc_fence_after();
            const uint32_t lane_off = (uint32_t)(q * 32) << 16;
            if (gate_up) {
                // tile-0 warps take tokens 0-63, tile-1 warps 64-127
                const int64_t i = r0 + r;
                for (int c0 = tile * 64; c0 < tile * 64 + 64; c0 += 32) {
                    float g[32], u[32];
                    tc_ld32(tmem_d + lane_off + c0, g);
                    tc_ld32(tmem_d + kQmmTok + lane_off + c0, u);
                    if (i < p.I)
                        for (int j = 0; j < 32; ++j) {
                            const int64_t m = m0 + c0 + j;
                            if (m < p.M)
                                p.y[m * p.I + i] = f32_to_bf16_bits(
                                    g[j] / (1.0f + __expf(-g[j])) * u[j]);
                        }
                }
            } else {
                int sidx = 0;
                if (p.mode == 1 && n >= 0)
                    while (sidx + 1 < p.nsec && n >= p.sec_start[sidx + 1])
                        ++sidx;
                for (int c0 = 0; c0 < kQmmTok; c0 += 32) {
                    float d[32];
                    tc_ld32(tmem_d + tile * kQmmTok + lane_off + c0, d);
                    if (n < 0) continue;
                    for (int j = 0; j < 32; ++j) {
                        const int64_t m = m0 + c0 + j;
                        if (m >= p.M) break;
                        if (p.mode == 0) {
                            p.y[m * p.N + n] = f32_to_bf16_bits(d[j]);
                        } else {
                            const int64_t jj = n - p.sec_start[sidx];
                            const int64_t size =
                                p.sec_start[sidx + 1] - p.sec_start[sidx];
                            float val = d[j];
                            if (p.sec_bias[sidx])
                                val += bf16_bits_to_f32(p.sec_bias[sidx][jj]);
                            p.sec_out[sidx][m * size + jj] = f32_to_bf16_bits(val);
                        }
                    }
                }
            }
        }
    }

    // ------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing may still be landing in shared memory or tensor memory
        for (int kb = s_xconsumed; kb < s_xissued; ++kb)
            if (!mbar_wait(&xfull[kb % kQmmXStages], (kb / kQmmXStages) & 1))
                break;
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

template <int BITS>
static int qmm_launch(const QmmArgs &a, unsigned char *ws, cudaStream_t st) {
    const int64_t M = a.M, K = a.w.K;
    const int64_t kext = qmm_kext(K);
    unsigned int *status = reinterpret_cast<unsigned int *>(ws);
    __half *xe = reinterpret_cast<__half *>(ws + kStatusBytes);

    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm status reset: %s",
                         cudaGetErrorString(e));
    const int64_t items = M * (K / 64);
    const int pthreads = 128;
    int64_t pblocks = (items + pthreads - 1) / pthreads;
    if (pblocks > (int64_t)num_sms() * 16) pblocks = (int64_t)num_sms() * 16;
    qmm_prepass_kernel<BITS><<<(unsigned)pblocks, pthreads, 0, st>>>(
        a.x, M, (int)K, kext, xe, status);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm pre-pass: %s", cudaGetErrorString(e));

    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode)
        return set_error(GWA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)kext, (cuuint64_t)M};
    const cuuint64_t gstride[1] = {(cuuint64_t)kext * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kQmmTok};
    const cuuint32_t estride[2] = {1, 1};
    CUresult cr = encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xe, gdim,
                         gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS)
        return set_error(GWA_ERR_CUDA, "tensor map encode failed (%d)", (int)cr);

    QmmParams p{};
    p.M = M;
    p.K = (int)K;
    p.kext = kext;
    p.nkb = (int)(kext / 64);
    p.G = (int)(K / 64);
    p.wq = a.w.wq;
    p.sc = a.w.scales;
    p.bi = a.w.biases;
    p.N = a.w.N;
    p.I = a.w.N / 2;
    p.mode = a.mode;
    p.y = a.y;
    p.nsec = a.nsec;
    for (int s = 0; s <= a.nsec && a.mode == 1; ++s) p.sec_start[s] = a.sec_start[s];
    for (int s = 0; s < a.nsec && a.mode == 1; ++s) {
        p.sec_out[s] = a.sec_out[s];
        p.sec_bias[s] = a.sec_bias[s];
    }
    p.status = status;

    auto kern = qmm_tc_kernel<BITS>;
    int dummy = 0;
    e = occupancy_grid(reinterpret_cast<const void *>(kern), kQmmThreads,
                       kQmmSmem, &dummy);
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm setup: %s", cudaGetErrorString(e));
    const int64_t rows = a.mode == 2 ? p.I : p.N;
    const int64_t per_cta = a.mode == 2 ? kQmmRows : 2 * kQmmRows;
    dim3 grid((unsigned)((rows + per_cta - 1) / per_cta),
              (unsigned)((M + kQmmTok - 1) / kQmmTok));
    kern<<<grid, kQmmThreads, kQmmSmem, st>>>(map, p);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return set_error(GWA_ERR_CUDA, "qmm launch: %s", cudaGetErrorString(e));
    return GWA_OK;
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
    return a.w.bits == 4 ? qmm_launch<4>(a, ws, st) : qmm_launch<8>(a, ws, st);
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
