// Dense decode kernels (M <= 8): plain quantized projection, fused
// projection written to separate section buffers, and fused gate+up with the
// SwiGLU epilogue.
//
//   qmv:       "Sanctum-MLX" (QuantizedLinear group_size=64) and "The
//              Cathedral Doubled Itself" (quantized_matmul).
//   sections:  "The Cathedral Doubled Itself", "The two fusions" (Phase 1A:
//              one matmul over [q_out + 2*kv_out, hidden/8], split on the
//              last axis) and "The trap that ate three hours" (each part must
//              be its own contiguous, offset-0 buffer).  Here the split costs
//              nothing: each output row is stored straight into its section.
//   gate+up:   same page, Phase 1B (gate_proj and up_proj before SiLU and the
//              multiply).  One warp owns gate rows n.. and up rows I+n.., so
//              SiLU(g)*u is formed in registers and only h is written.
//
// Grid: persistent-style.  Warp-block b (R rows) runs on CTA b % grid, so the
// blocks spread evenly over the SMs whatever N is.
#include "internal.h"
#include "qmv_dense.cuh"

namespace gwa {

enum DenseMode { kPlain = 0, kSections = 1, kGateUp = 2, kRope = 3 };

// kRope: QKV sections with the rotary embedding, pairs of rows (i, i + d/2)
// of a head (rope_pair_row) laid out like gate/up pairs.

template <int BITS, int MT, int R, int MODE>
__global__ void __launch_bounds__(kDenseThreads)
    qmv_dense_kernel(DenseParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int tok[8];
    __shared__ int s_mk;  // some staged group is marked (common.cuh)
    if (threadIdx.x < 8)
        tok[threadIdx.x] = (int)threadIdx.x < p.M ? (int)threadIdx.x : -1;
    if (threadIdx.x == 0) s_mk = 0;
    __syncthreads();
    stage_x<BITS>(p.x, p.K, tok, MT, p.nch, smem, &s_mk);
    __syncthreads();
    const bool mk = s_mk != 0;

    const int lane = threadIdx.x & (kWarp - 1);
    const int warp = threadIdx.x / kWarp;
    const WView v{reinterpret_cast<const uint4 *>(p.wq), p.sc, p.bi, p.nch,
                  p.G};
    constexpr bool PAIRS = MODE == kGateUp || MODE == kRope;
    constexpr int RP = PAIRS ? R / 2 : R;  // output units per block

    for (int64_t b = blockIdx.x + (int64_t)gridDim.x * warp; b < p.nblocks;
         b += (int64_t)gridDim.x * (kDenseThreads / kWarp)) {
        int64_t rows[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if constexpr (MODE == kGateUp) {
                const int64_t n = b * RP + (r % RP);
                rows[r] = n < p.I ? (r < RP ? n : p.I + n) : -1;
            } else if constexpr (MODE == kRope) {
                const int64_t n = b * RP + (r % RP);  // pair
                rows[r] = n < p.N / 2 ? rope_pair_row(n, r / RP, p.rope_hd) : -1;
            } else {
                const int64_t n = b * R + r;
                rows[r] = n < p.N ? n : -1;
            }
        }
        int midx[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) midx[m] = m;
        float acc[R][MT];
        if (mk)
            rows_dot<BITS, MT, R, true>(v, rows, midx, MT, smem, lane, acc);
        else
            rows_dot<BITS, MT, R, false>(v, rows, midx, MT, smem, lane, acc);
        warp_reduce<R, MT>(acc);

#pragma unroll
        for (int r = 0; r < RP; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (lane != r * MT + m || m >= p.M) continue;
                const int64_t n = PAIRS ? b * RP + r : rows[r];
                if (n < 0 || (MODE == kGateUp && n >= p.I) ||
                    (MODE == kRope && n >= p.N / 2))
                    continue;
                if constexpr (MODE == kRope) {
                    // pair n: rows r0 and r0 + d/2 of one head; sections
                    // are whole heads
                    const int half = p.rope_hd / 2;
                    const int64_t r0 = rope_pair_row(n, 0, p.rope_hd);
                    int s = 0;
                    while (s + 1 < p.nsec && r0 >= p.sec_start[s + 1]) ++s;
                    const int64_t j = r0 - p.sec_start[s];
                    const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
                    float a = acc[r][m], c = acc[RP + r][m];
                    if (p.sec_bias[s]) {
                        a += bf16_bits_to_f32(p.sec_bias[s][j]);
                        c += bf16_bits_to_f32(p.sec_bias[s][j + half]);
                    }
                    if (r0 < p.rope_end) {
                        const float2 t = p.rope_cs[(int64_t)m * half + n % half];
                        const float a2 = a * t.x - c * t.y;
                        c = c * t.x + a * t.y;
                        a = a2;
                    }
                    uint16_t *o = p.sec_out[s] + (int64_t)m * size + j;
                    o[0] = f32_to_bf16_bits(a);
                    o[half] = f32_to_bf16_bits(c);
                } else if constexpr (MODE == kPlain) {
                    p.y[(int64_t)m * p.N + n] = f32_to_bf16_bits(acc[r][m]);
                } else if constexpr (MODE == kGateUp) {
                    p.y[(int64_t)m * p.I + n] =
                        f32_to_bf16_bits(silu_mul(acc[r][m], acc[RP + r][m]));
                } else {
                    int s = 0;
                    while (s + 1 < p.nsec && n >= p.sec_start[s + 1]) ++s;
                    const int64_t j = n - p.sec_start[s];
                    const int64_t size = p.sec_start[s + 1] - p.sec_start[s];
                    float val = acc[r][m];
                    if (p.sec_bias[s]) val += bf16_bits_to_f32(p.sec_bias[s][j]);
                    p.sec_out[s][(int64_t)m * size + j] = f32_to_bf16_bits(val);
                }
            }
    }
}

// ------------------------------------------------------------ host side
template <int BITS, int MT, int R, int MODE>
static cudaError_t launch_dense_t(const DenseParams &p, cudaStream_t st) {
    auto kern = qmv_dense_kernel<BITS, MT, R, MODE>;
    const size_t smem = XStage<BITS>::bytes(MT, p.nch);
    int grid = 0;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   kDenseThreads, smem, &grid);
    if (e != cudaSuccess) return e;
    DenseParams q = p;
    q.nblocks = MODE == kGateUp ? (p.I + R / 2 - 1) / (R / 2)
                : MODE == kRope ? (p.N / 2 + R / 2 - 1) / (R / 2)
                                : (p.N + R - 1) / R;
    if ((int64_t)grid > q.nblocks) grid = (int)q.nblocks;
    if (grid < 1) grid = 1;
    kern<<<grid, kDenseThreads, smem, st>>>(q);
    return cudaGetLastError();
}

template <int BITS, int MODE>
static cudaError_t launch_dense_m(const DenseParams &p, cudaStream_t st) {
    // gate+up uses R/2 gate rows + R/2 up rows per warp block
    if (p.M <= 1) return launch_dense_t<BITS, 1, 4, MODE>(p, st);
    if (p.M <= 2) return launch_dense_t<BITS, 2, 4, MODE>(p, st);
    if (p.M <= 4) return launch_dense_t<BITS, 4, 4, MODE>(p, st);
    return launch_dense_t<BITS, 8, 2, MODE>(p, st);
}

// Largest token count per launch whose staged activations fit in shared
// memory.
int dense_max_tokens(int bits, int nch) {
    const size_t cap = kMaxDynSmem;
    int mt = 8;
    while (mt > 1 && (bits == 4 ? XStage<4>::bytes(mt, nch)
                                : XStage<8>::bytes(mt, nch)) > cap)
        mt /= 2;
    const size_t one = bits == 4 ? XStage<4>::bytes(1, nch)
                                 : XStage<8>::bytes(1, nch);
    return one > cap ? 0 : mt;
}

cudaError_t launch_dense(int mode, const DenseParams &p, cudaStream_t st) {
    if (mode == kRope)
        return p.bits == 4 ? launch_dense_m<4, kRope>(p, st)
                           : launch_dense_m<8, kRope>(p, st);
    if (p.bits == 4) {
        if (mode == kPlain) return launch_dense_m<4, kPlain>(p, st);
        if (mode == kSections) return launch_dense_m<4, kSections>(p, st);
        return launch_dense_m<4, kGateUp>(p, st);
    }
    if (mode == kPlain) return launch_dense_m<8, kPlain>(p, st);
    if (mode == kSections) return launch_dense_m<8, kSections>(p, st);
    return launch_dense_m<8, kGateUp>(p, st);
}

}  // namespace gwa
