// Affine group quantization of bf16 weights: the requantize step of
// "Sanctum-MLX", "The April 2026 cutover" (LoRA merge at load dequantizes,
// adds the delta and requantizes at group size 64; "File map": lora.rs also
// merges the switch_mlp expert weights).  The pages state no rule; the
// reading used here, per group of 64 consecutive inputs of a row:
//
//   scale = bf16_rn((max - min) / (2^b - 1)),  bias = min (a bf16 already;
//   a zero minimum is stored as +0),
//   code  = clamp(rint((w - bias) / scale), 0, 2^b - 1), or 0 if scale == 0,
//
// in IEEE fp32 (correctly rounded divide, round half to even), codes packed
// lowest bits first.  Finite inputs only.
//
// Eight lanes share a group: each loads 16 bytes (eight inputs), the lanes
// agree on the minimum and maximum with three shuffles, and each packs its
// eight codes into one (u4) or two (u8) words; the group's first lane writes
// the scale and bias.  A warp covers four consecutive groups per step, so
// its loads are 512 contiguous bytes.  The HBM floor is 2 bytes read and
// b/8 + 1/16 written per weight (~54 us for a 27648 x 5120 u4 weight), but
// the exactly rounded codes take ~10 instructions per weight, so the kernel
// runs at about a third of HBM bandwidth, limited by instruction issue
// (issuing four steps' loads ahead changed nothing).
#include "common.cuh"
#include "internal.h"

namespace gwa {

template <int BITS>
__global__ void __launch_bounds__(256)
    quantize_affine_kernel(const uint16_t *__restrict__ w, int64_t groups,
                           uint32_t *__restrict__ wq, uint16_t *__restrict__ sc,
                           uint16_t *__restrict__ bi) {
    constexpr uint32_t QMAX = (1u << BITS) - 1u;
    const int lane = threadIdx.x & (kWarp - 1);
    const int sub = lane >> 3, l8 = lane & 7;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / kWarp;
    // every lane of a warp takes the same trip count (the shuffles need all
    // 32); groups past the end compute on zeros and store nothing
    for (int64_t q4 = warp * 4; q4 < groups; q4 += nwarps * 4) {
        const int64_t g = q4 + sub;
        const bool live = g < groups;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (live)
            u = reinterpret_cast<const uint4 *>(w)[g * 8 + l8];
        float v[8];
        v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
        v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
        v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
        float lo = v[0], hi = v[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            lo = fminf(lo, v[i]);
            hi = fmaxf(hi, v[i]);
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, m));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, m));
        }
        lo = lo + 0.0f;  // a zero minimum is stored as +0
        const uint16_t sbits =
            f32_to_bf16_bits(__fdiv_rn(hi - lo, (float)QMAX));
        const float s = bf16_bits_to_f32(sbits);
        // The code is rint of the correctly rounded quotient d / s.  A
        // product with the correctly rounded reciprocal is within
        // 1.5 * 2^-23 * d/s (<= 4.6e-5, d/s <= ~257) of that quotient, so its
        // rounding can differ only when it lies within that distance of a
        // half-integer (about one input in 10^4); a lane holding such an
        // input redoes its eight codes by the division, which gives the same
        // codes for the others.  Subnormal scales (a reciprocal that may
        // overflow) always divide.
        const bool fast = s >= 1.17549435e-38f;
        const float r = fast ? __frcp_rn(s) : 0.0f;
        uint32_t q[8];
        float emax = 0.0f;  // the largest distance of a product from an integer
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float d = v[i] - lo;  // >= 0, as in the reading
            const float t = d * r;
            // t + 1.5 * 2^23 rounds t to an integer, ties to even, into
            // the low mantissa bits (0 <= t < 2^22)
            const float tt = t + 12582912.0f;
            emax = fmaxf(emax, fabsf(t - (tt - 12582912.0f)));
            q[i] = min(__float_as_uint(tt) - 0x4b400000u, QMAX);
        }
        // a product within reach of a half-integer, or no usable reciprocal:
        // all eight codes again by the division (rare; uniform per lane)
        if (!fast || emax > 0.5f - 0x1p-12f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float d = v[i] - lo;
                uint32_t c = 0u;
                if (s != 0.0f) {
                    const float tx = rintf(__fdiv_rn(d, s));
                    c = tx <= 0.0f ? 0u : tx >= (float)QMAX ? QMAX : (uint32_t)tx;
                }
                q[i] = c;
            }
        }
        if (!live) continue;
        if constexpr (BITS == 4) {
            uint32_t word = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) word |= q[i] << (4 * i);
            wq[g * 8 + l8] = word;
        } else {
            const uint32_t w0 = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
            const uint32_t w1 = q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24);
            reinterpret_cast<uint2 *>(wq)[g * 8 + l8] = make_uint2(w0, w1);
        }
        if (l8 == 0) {
            sc[g] = sbits;
            bi[g] = (uint16_t)(__float_as_uint(lo) >> 16);
        }
    }
}

cudaError_t launch_quantize(const uint16_t *w, int64_t N, int64_t K, int bits,
                            uint32_t *wq, uint16_t *sc, uint16_t *bi,
                            cudaStream_t st) {
    const int64_t groups = N * (K / kGroup);
    if (groups == 0) return cudaSuccess;
    constexpr int kThreads = 256;  // 8 warps: 32 groups per block and step
    int64_t blocks = (groups + 31) / 32;
    const int64_t cap = (int64_t)num_sms() * 8;  // 2048 threads per SM
    if (blocks > cap) blocks = cap;
    if (bits == 4)
        quantize_affine_kernel<4><<<(unsigned)blocks, kThreads, 0, st>>>(
            w, groups, wq, sc, bi);
    else
        quantize_affine_kernel<8><<<(unsigned)blocks, kThreads, 0, st>>>(
            w, groups, wq, sc, bi);
    return cudaGetLastError();
}

}  // namespace gwa
