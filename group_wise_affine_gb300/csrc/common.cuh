// Device helpers shared by the decode (GEMV) kernels.
//
// Packed layout (MLX affine integer weights, "saragossa", "Quantization
// formats"; "The Cathedral Doubled Itself", "The two fusions"): a row of K
// inputs is K*bits/32 uint32 words, code k mod P of word k/P at bits
// [bits*(k mod P), +bits), lowest bits first.  One bf16 scale and one bf16
// bias per 64 inputs: w = scale*q + bias.
//
// Exact code -> fp32 conversion without an int->float instruction: OR the
// code into the mantissa of a power of two.  A 4-bit code placed at mantissa
// bits [15,19) under exponent 2^8 reads as 256 + q; placed at bits [19,23)
// under exponent 2^4 it reads as 16 + q.  One shift of the packed word lines
// up two codes at once (one in each window), so eight codes cost four shifts
// and eight AND-OR (LOP3) operations and land as four fp32 pairs that feed
// packed fp32x2 FMAs.  The constants are removed once per chunk:
//   sum_k x_k (C_k + q_k) = sum_k x_k q_k + sum_k C_k x_k,
// with sum_k C_k x_k precomputed per chunk of activations.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gwa {

constexpr int kGroup = 64;
constexpr int kWarp = 32;

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
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

// ---------------------------------------------------------------- u4
// Constants the magic windows add, per code position inside a word:
// odd positions read as 256 + q, even positions as 16 + q.
constexpr float kU4Odd = 256.0f;
constexpr float kU4Even = 16.0f;

// Eight 4-bit codes of one word -> four pairs (odd-position value,
// even-position value):
//   p[0] = (256+q3, 16+q4)   p[1] = (256+q5, 16+q6)
//   p[2] = (256+q1, 16+q2)   p[3] = (256+q7, 16+q0)
// Activations are stored in the matching order x3 x4 x5 x6 | x1 x2 x7 x0.
__device__ __forceinline__ void unpack_u4(uint32_t w, float2 (&p)[4]) {
    const uint32_t lo_mask = 0x00078000u, lo_magic = 0x43800000u;  // 2^8
    const uint32_t hi_mask = 0x00780000u, hi_magic = 0x41800000u;  // 2^4
    uint32_t t0 = w << 3;                       // q3 -> [15,19), q4 -> [19,23)
    uint32_t t1 = w >> 5;                       // q5, q6
    uint32_t t2 = w << 11;                      // q1, q2
    uint32_t t3 = __funnelshift_l(w, w, 19);    // q7 -> [15,19), q0 -> [19,23)
    p[0] = make_float2(__uint_as_float((t0 & lo_mask) | lo_magic),
                       __uint_as_float((t0 & hi_mask) | hi_magic));
    p[1] = make_float2(__uint_as_float((t1 & lo_mask) | lo_magic),
                       __uint_as_float((t1 & hi_mask) | hi_magic));
    p[2] = make_float2(__uint_as_float((t2 & lo_mask) | lo_magic),
                       __uint_as_float((t2 & hi_mask) | hi_magic));
    p[3] = make_float2(__uint_as_float((t3 & lo_mask) | lo_magic),
                       __uint_as_float((t3 & hi_mask) | hi_magic));
}
// Position of the activation that pairs with slot i of the unpacked word.
__device__ __forceinline__ int u4_perm(int i) {
    // x3 x4 x5 x6 x1 x2 x7 x0
    return (0x07216543 >> (4 * i)) & 0xf;
}

// ---------------------------------------------------------------- u8
constexpr float kU8Const = 256.0f;

// Four 8-bit codes of one word -> two pairs (256+q0, 256+q1), (256+q2, 256+q3).
__device__ __forceinline__ void unpack_u8(uint32_t w, float2 (&p)[2]) {
    const uint32_t mask = 0x007f8000u, magic = 0x43800000u;  // [15,23), 2^8
    p[0] = make_float2(__uint_as_float(((w << 15) & mask) | magic),
                       __uint_as_float(((w << 7) & mask) | magic));
    p[1] = make_float2(__uint_as_float(((w >> 1) & mask) | magic),
                       __uint_as_float(((w >> 9) & mask) | magic));
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
