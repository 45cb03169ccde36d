// Device helpers shared by the kernels: bf16 conversions, the integer dot
// used by the decode kernels, and mbarrier / bulk-copy / PDL wrappers.
//
// Packed layout (MLX affine integer weights, "saragossa", "Quantization
// formats"; "The Cathedral Doubled Itself", "The two fusions"): a row of K
// inputs is K*bits/32 uint32 words, code k mod P of word k/P at bits
// [bits*(k mod P), +bits), lowest bits first.  One bf16 scale and one bf16
// bias per 64 inputs: w = scale*q + bias.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gwa {

constexpr int kGroup = 64;
constexpr int kWarp = 32;

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) * 65536u);
}
// The two bf16 halves of a 32-bit word, widened exactly.
__device__ __forceinline__ float bf16_lo(uint32_t v) {
    return __uint_as_float(v << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t v) {
    return __uint_as_float(v & 0xffff0000u);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// The OCP FP8 E4M3 number of the low byte of `code` (fp8 weights): the
// hardware conversion to fp16, which holds every E4M3 value exactly
// (subnormals and NaN included), then to fp32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(
        static_cast<__nv_fp8_storage_t>(code & 0xffu), __NV_E4M3);
    return __half2float(__half(h));
}

// 16-byte streaming load of packed weights: read once, keep out of L1.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_u16(const uint16_t *p) {
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

template <int BITS>
struct Fmt;
template <>
struct Fmt<4> {
    static constexpr int kCodesPerWord = 8;
    static constexpr int kChunkCodes = 32;  // one 16-byte chunk
};
template <>
struct Fmt<8> {
    static constexpr int kCodesPerWord = 4;
    static constexpr int kChunkCodes = 16;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace gwa

// ---------------------------------------------------------------- integer dot
namespace gwa {
// The decode kernels form each group's sum of code x activation as an exact
// integer.  Activations are encoded per group of 64 as int16 with a
// power-of-two scale 2^E chosen from the group's largest exponent (the
// largest magnitude maps into [2^14, 2^15)).  A bf16 value carries 8
// significant bits, so every value within 2^7 of the group's largest
// exponent is represented exactly; smaller ones round to the group's quantum
// (at most 2^-15 of the largest magnitude; groups where that matters take
// an fp32 path, see "marked groups" below).  Codes stay unsigned bytes, and
// dp2a forms two 16x8-bit products per instruction into an int32 (at most
// 64 * 255 * 32640 < 2^31 per group).  Per group:
//   y += (scale * 2^E) * D + bias * sum_k x_k,   D = sum_k q_k * xi_k.
__device__ __forceinline__ int dp2a_lo(uint32_t a16, uint32_t b8, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a16), "r"(b8), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a16, uint32_t b8, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a16), "r"(b8), "r"(c));
    return d;
}
// Four unsigned code bytes times four signed bytes (a residual plane, see
// "marked groups"), added to c.
__device__ __forceinline__ int dp4a_us(uint32_t a8, uint32_t b8, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a8), "r"(b8), "r"(c));
    return d;
}

// Exponent field (biased, 0..255) of an fp32 value.
__device__ __forceinline__ int f32_exp_field(float v) {
    return (int)((__float_as_uint(v) >> 23) & 0xffu);
}

// Scale of a group whose largest exponent field is ef: f = 2^E and 1/f.
// Groups whose magnitudes all lie below 2^-112 are encoded as zero (their
// contribution is below 64 * 2^-112 * |w|); their plain sum still feeds the
// bias term.
__device__ __forceinline__ void group_scale(int ef, float &f, float &finv) {
    if (ef < 15) {
        f = 0.f;
        finv = 0.f;
    } else {
        f = __uint_as_float((uint32_t)(ef - 14) << 23);      // 2^(ef-141)
        finv = __uint_as_float((uint32_t)(268 - ef) << 23);  // 2^(141-ef)
    }
}

// int16 pair (lo = a, hi = b) of two activations already multiplied by 1/f.
__device__ __forceinline__ uint32_t i16_pair(float a, float b) {
    return ((uint32_t)__float2int_rn(a) & 0xffffu) |
           ((uint32_t)__float2int_rn(b) << 16);
}

// u4: the four int16 pairs of one word's activations, in dp2a order:
//   (x0,x2) (x4,x6) (x1,x3) (x5,x7)  [x scaled by finv]
__device__ __forceinline__ void u4_pairs(const float *v, float finv,
                                         uint32_t (&pr)[4]) {
    pr[0] = i16_pair(v[0] * finv, v[2] * finv);
    pr[1] = i16_pair(v[4] * finv, v[6] * finv);
    pr[2] = i16_pair(v[1] * finv, v[3] * finv);
    pr[3] = i16_pair(v[5] * finv, v[7] * finv);
}
// u8: the two pairs of one word: (x0,x1) (x2,x3).
__device__ __forceinline__ void u8_pairs(const float *v, float finv,
                                         uint32_t (&pr)[2]) {
    pr[0] = i16_pair(v[0] * finv, v[1] * finv);
    pr[1] = i16_pair(v[2] * finv, v[3] * finv);
}

// Integer dot of one packed word with its activation pairs, into two
// accumulators.  u4: the low nibbles (q0 q2 q4 q6) go to acc[0]; the high
// nibbles stay in place as 16*q (q1 q3 q5 q7, no shift needed) and go to
// acc[1], which therefore holds 16x its sum, exactly (at most
// 32 * 240 * 32640 < 2^31 per chunk).  Combine with dot_total.
__device__ __forceinline__ void word_dot_u4(uint32_t w, const uint32_t *pr,
                                            int (&acc)[2]) {
    const uint32_t lo = w & 0x0f0f0f0fu;
    const uint32_t hi = w & 0xf0f0f0f0u;
    acc[0] = dp2a_hi(pr[1], lo, dp2a_lo(pr[0], lo, acc[0]));
    acc[1] = dp2a_hi(pr[3], hi, dp2a_lo(pr[2], hi, acc[1]));
}
__device__ __forceinline__ void word_dot_u8(uint32_t w, const uint32_t *pr,
                                            int (&acc)[2]) {
    acc[0] = dp2a_lo(pr[0], w, acc[0]);
    acc[1] = dp2a_hi(pr[1], w, acc[1]);
}
template <int BITS>
__device__ __forceinline__ int dot_total(const int (&acc)[2]) {
    return BITS == 4 ? acc[0] + (acc[1] >> 4) : acc[0] + acc[1];
}

// ------------------------------------------------------- marked groups
// The one-plane encoding above is exact when a group's values lie within
// 2^7 of its largest one; smaller values round to the group's quantum f.
// One large activation among ordinary ones (an outlier channel), or values
// spread over many binades (a gated product such as SiLU(g) * u), then
// round many values of the group, and an output whose products cancel loses
// more than the fp32 sum it stands for.  So every encoder also forms, per
// group and in units of f,
//   R = sum_k |x_k / f - xi_k|   (the rounding error, exact term by term)
//   A = sum_k |x_k| / f,
// and marks the group when R > 2^-16 * A (an unmarked group thus has
// sum_k |x_k - f * xi_k| <= 2^-16 * sum_k |x_k|, 128 times less than
// rounding its activations to bf16 once more).  Measured on 20000 groups:
// N(0,1) activations reach R / A = 2^-16.9 at most (none marked), Laplace
// ones mark 0.09% of groups, SiLU(g) * u with g, u ~ N(0,1) 18%, and one
// value 30 times the rest of its group, or magnitudes spread over 2^20,
// mark it.  A marked group is finished one of two ways:
//  * two planes (the one- and few-token decode kernels): the int16 image
//    stays, and the lane adds a second dot with the int8 residual plane
//    lo_k = rint(2^7 * (x_k / f - xi_k)) (dp4a, four products per
//    instruction): the rounding error drops below 2^-8 f per value, so
//    R <= 0.25 and, as A >= 2^14 always, R <= 2^-16 * A for every input;
//  * fp32 (the other kernels): the group keeps its raw bf16 activations in
//    the slots of its int16 pairs (same size, same pair order), its stored
//    scale is negative, and its dots are taken by the fp32 counterparts of
//    dp2a below (codes and activations exact, every product exact, fp32
//    sums).
// The kernels decide before their main loop, per CTA (one-token, staged,
// general and MoE kernels) or per warp (streaming kernel), whether any
// group is marked, and otherwise run a copy of the loop without the marked
// path.
__device__ __forceinline__ bool group_marked(float r, float a) {
    return r * 65536.0f > a;
}

// |v * finv - rint(v * finv)|, exact: v is a bf16 value and finv a power of
// two, so v * finv is exact; adding 1.5 * 2^23 rounds it to the integer the
// encoders store (half to even), and the difference has no more bits than v.
__device__ __forceinline__ float i16_resid(float v, float finv) {
    const float t = fmaf(v, finv, 12582912.0f) - 12582912.0f;
    return fabsf(fmaf(v, finv, -t));
}

// Signed 2^7 * (v * finv - rint(v * finv)) rounded to an integer in
// [-64, 64], as the low byte of the result (two's complement): one entry
// of a residual plane.  Both roundings are half to even.
__device__ __forceinline__ uint32_t i8_resid(float v, float finv) {
    const float t = fmaf(v, finv, 12582912.0f) - 12582912.0f;
    const float r = fmaf(v, finv, -t);  // exact, in [-0.5, 0.5]
    return __float_as_uint(fmaf(r, 128.0f, 12582912.0f)) & 0xffu;
}

// The raw bf16 pair (lo = a, hi = b) of two values widened from bf16.
__device__ __forceinline__ uint32_t raw_pair(float a, float b) {
    return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
}

// Byte I of b as an exact fp32 value: the permute builds 2^23 + byte, and
// subtracting 2^23 is exact.
template <int I>
__device__ __forceinline__ float byte_f32(uint32_t b) {
    return __uint_as_float(__byte_perm(b, 0x4b000000u, 0x7440 | I)) - 8388608.0f;
}

// fp32 counterparts of dp2a_lo / dp2a_hi for a marked group: a holds two raw
// bf16 activations, b the code bytes; every product is exact (8 by 8
// significant bits), the sums round in fp32.
__device__ __forceinline__ float fdp2a_lo(uint32_t a, uint32_t b, float c) {
    return fmaf(bf16_hi(a), byte_f32<1>(b), fmaf(bf16_lo(a), byte_f32<0>(b), c));
}
__device__ __forceinline__ float fdp2a_hi(uint32_t a, uint32_t b, float c) {
    return fmaf(bf16_hi(a), byte_f32<3>(b), fmaf(bf16_lo(a), byte_f32<2>(b), c));
}

// word_dot_u4 / word_dot_u8 and dot_total in fp32 (one chunk word at a
// time): the true sum of q_k * x_k, the u4 high nibbles' 16x divided out.
__device__ __forceinline__ void fword_dot_u4(uint32_t w, const uint32_t *pr,
                                             float (&acc)[2]) {
    const uint32_t lo = w & 0x0f0f0f0fu;
    const uint32_t hi = w & 0xf0f0f0f0u;
    acc[0] = fdp2a_hi(pr[1], lo, fdp2a_lo(pr[0], lo, acc[0]));
    acc[1] = fdp2a_hi(pr[3], hi, fdp2a_lo(pr[2], hi, acc[1]));
}
__device__ __forceinline__ void fword_dot_u8(uint32_t w, const uint32_t *pr,
                                             float (&acc)[2]) {
    acc[0] = fdp2a_lo(pr[0], w, acc[0]);
    acc[1] = fdp2a_hi(pr[1], w, acc[1]);
}
template <int BITS>
__device__ __forceinline__ float fdot_total(const float (&acc)[2]) {
    return BITS == 4 ? fmaf(acc[1], 0.0625f, acc[0]) : acc[0] + acc[1];
}

// Element i (a run-time index) of a register array, by a chain of selects
// (no local-memory indexing); used by the marked paths, which run one row at
// a time so that their registers stay few.
template <typename T, int N>
__device__ __forceinline__ T pick(const T (&a)[N], int i) {
    T v = a[0];
#pragma unroll
    for (int k = 1; k < N; ++k)
        if (i == k) v = a[k];
    return v;
}

// sum_k q_k * x_k of one 16-byte chunk word by word (fword_dot_*), w the
// chunk's four code words and pr its activation pairs (4 per word for u4, 2
// for u8) as raw bf16: a marked chunk's dot in fp32.  One word per loop
// step, so that only that word's products are in flight.
template <int BITS>
__device__ __forceinline__ float chunk_dot_f32(const uint4 &w,
                                               const uint32_t (&pr)[BITS == 4 ? 16 : 8]) {
    constexpr int P = BITS == 4 ? 4 : 2;
    float a[2] = {0.f, 0.f};
#pragma unroll 1
    for (int wd = 0; wd < 4; ++wd) {
        const uint32_t word = wd == 0 ? w.x : wd == 1 ? w.y : wd == 2 ? w.z : w.w;
        uint32_t p[P];
#pragma unroll
        for (int i = 0; i < P; ++i) {
            p[i] = pr[i];
#pragma unroll
            for (int k = 1; k < 4; ++k)
                if (wd == k) p[i] = pr[k * P + i];
        }
        if constexpr (BITS == 4)
            fword_dot_u4(word, p, a);
        else
            fword_dot_u8(word, p, a);
    }
    return fdot_total<BITS>(a);
}

}  // namespace gwa

// ---------------------------------------------------------------- async copy
// mbarrier + bulk-copy helpers (sm_90+ PTX).  Every wait is bounded by the
// global timer: after kWaitLimitNs the wait gives up and reports failure, so
// a broken pipeline returns an error instead of hanging the GPU.
namespace gwa {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete; false after the time limit.
__device__ __forceinline__ bool mbar_wait(
    uint64_t *bar, uint32_t parity,
    unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// The same wait with a suspend-time hint: a thread whose phase is not yet
// complete sleeps (up to `hint_ns`, woken early when the phase completes)
// instead of polling, which leaves the issue slots to the working warps.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar,
                                                    uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(
    uint64_t *bar, uint32_t parity,
    unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity, 1000000u))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// Rotary embedding pairs: unit u is the pair of rows (i, i + d/2) of head
// u / (d/2), i = u mod d/2; row of half h (0 or 1).  The projections lay such
// a pair out like a gate/up pair (pairs < 2^31: rows < 2^30).
__device__ __forceinline__ int64_t rope_pair_row(int64_t u, int h, int d) {
    const int half = d / 2, uu = (int)u;
    return (int64_t)(uu / half) * d + (uu % half) + h * half;
}

// cos and sin of the rotary angle theta = pos * base^(-2i/d) (textbook
// RoPE, pair index i of a head of d), given r = base^(-2/d) in fp64:
// base^(-2i/d) = r^i by repeated squaring (a dozen fp64 products; relative
// error ~1e-15), and theta is reduced modulo 2 pi in fp64 (2 pi split in two
// doubles), so the fp32 sincos sees an argument within [-pi, pi] accurate to
// ~1e-14 even at positions of 10^5 and more.  An fp32 angle would be off by
// ~1e-2 rad at position 32K; an fp64 pow per angle costs several times more
// on this GPU, whose fp64 rate is low.
__device__ __forceinline__ float2 rope_cos_sin(int pos, int i, double r) {
    double f = 1.0, b = r;
    for (int e = i; e > 0; e >>= 1) {
        if (e & 1) f *= b;
        b *= b;
    }
    const double theta = (double)pos * f;
    const double k = rint(theta * 0.15915494309189535);  // 1 / (2 pi)
    double t = fma(-k, 6.283185307179586, theta);
    t = fma(-k, 2.4492935982947064e-16, t);
    float sn, cs;
    sincosf((float)t, &sn, &cs);
    return make_float2(cs, sn);
}

// Contiguous global -> shared copy completing on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src,
                                         uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Recursive-halving transpose reduction of V values (V a power of two, at
// most 32) across the 32 lanes of a warp.  Afterwards lane l holds the
// warp-wide sum of value index (l >> (5 - log2 V)), and lanes whose low
// (5 - log2 V) bits are zero hold each index once.  Costs 31 shuffles in
// total for V = 32 instead of 5 per value.
template <int V>
__device__ __forceinline__ float transpose_reduce(float (&v)[V], int lane) {
    static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V");
#pragma unroll
    for (int half = V / 2, bit = 16; half >= 1; half /= 2, bit /= 2) {
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
    for (int bit = 16 / V; bit >= 1; bit /= 2)
        r += __shfl_xor_sync(0xffffffffu, r, bit);
    return r;
}

}  // namespace gwa
