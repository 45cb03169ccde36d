// Top-k MoE expert GEMV over stacked expert weights ("Sanctum-MLX": 3-D
// switch_mlp expert grids; "Four Candles For The Cathedral", "What's not in
// this batch": routed experts with per-expert gate_proj / up_proj, and the
// 6x regression that came from duplicating expert weights).  No weight is
// copied or duplicated here: the kernels read the caller's stacked tensor in
// place, and every distinct expert id of the call is streamed once.
//
// Gate+up mode: grid (pair blocks, slots).  The CTA of slot s owns expert
// e = ids[s] only if s is the first slot naming e; it then gathers every slot
// naming e (1 or 2 at decode batch sizes), stages those tokens and runs the
// fused gate+up row dots with the SiLU(g)*u epilogue.  Other CTAs of e exit.
//
// Down mode: grid over output-row blocks.  Each CTA stages every slot's input
// once, groups the slots by expert in first-occurrence order (in parallel, no
// scratch), then each lane walks (expert, chunk) items with a ring of
// prefetched loads, accumulating route_w * (W[e] h) per token in registers.
// The combine over experts is a register and warp-shuffle sum, so the output
// is written once, in bf16, with no atomics and no fp32 scratch.
#include "internal.h"
#include "qmv_dense.cuh"

namespace gwa {

constexpr int kMoeThreads = 256;
constexpr int kMoeDownThreads = 256;
constexpr int kMoeMaxSlots = 256;
constexpr int kMoeRP = 2;  // gate/up row pairs per warp

// ------------------------------------------------------------ gate + up
template <int BITS, int MT>
__device__ __forceinline__ void moe_gate_up_body(const MoeParams &p,
                                                 const WView &v,
                                                 const int *list, int mt,
                                                 int64_t i0,
                                                 const unsigned char *xs,
                                                 bool mk) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t I = p.N / 2;
    constexpr int R = 2 * kMoeRP;
    int64_t rows[R];
    const int64_t n0 = i0 + (int64_t)warp * kMoeRP;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t n = n0 + (r % kMoeRP);
        rows[r] = n < I ? (r < kMoeRP ? n : I + n) : -1;
    }
    int midx[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) midx[m] = m;
    float acc[R][MT];
    if (mk)
        rows_dot<BITS, MT, R, true>(v, rows, midx, MT, xs, lane, acc);
    else
        rows_dot<BITS, MT, R, false>(v, rows, midx, MT, xs, lane, acc);
    warp_reduce<R, MT>(acc);
#pragma unroll
    for (int r = 0; r < kMoeRP; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int64_t n = n0 + r;
            if (lane != r * MT + m || m >= mt || n >= I) continue;
            p.out[(int64_t)list[m] * I + n] =
                f32_to_bf16_bits(silu_mul(acc[r][m], acc[kMoeRP + r][m]));
        }
}

template <int BITS>
__global__ void __launch_bounds__(kMoeThreads)
    moe_gate_up_kernel(MoeParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int list[kMoeMaxSlots];
    __shared__ int tok[8];
    __shared__ int s_cnt, s_state;
    __shared__ int s_mk;  // some staged group of the pass is marked
    const int S = p.M * p.topk;
    const int slot = blockIdx.y;
    const int64_t I = p.N / 2;
    constexpr int kPairsPerCta = (kMoeThreads / 32) * kMoeRP;
    const int64_t i0 = (int64_t)blockIdx.x * kPairsPerCta;

    if (threadIdx.x == 0) {
        const int e = p.ids[slot];
        int state = 0, cnt = 0;
        if (e < 0 || e >= p.E) {
            state = 2;
            if (p.status && blockIdx.x == 0) atomicOr(p.status, 1);
        } else {
            for (int s = 0; s < slot; ++s)
                if (p.ids[s] == e) {
                    state = 1;
                    break;
                }
            if (!state)
                for (int s = slot; s < S; ++s)
                    if (p.ids[s] == e) list[cnt++] = s;
        }
        s_cnt = cnt;
        s_state = state;
    }
    __syncthreads();
    if (s_state == 1) return;  // another CTA owns this expert
    if (s_state == 2) {        // invalid id: this slot's outputs are zero
        for (int64_t i = i0 + threadIdx.x; i < i0 + kPairsPerCta && i < I;
             i += blockDim.x)
            p.out[(int64_t)slot * I + i] = 0;
        return;
    }
    const int64_t e = p.ids[slot];
    const WView v{reinterpret_cast<const uint4 *>(p.wq) + e * p.N * p.nch,
                  p.sc + e * p.N * p.G, p.bi + e * p.N * p.G, p.nch, p.G};
    const int cnt = s_cnt;
    // tokens of this expert in passes of at most four
    for (int base = 0; base < cnt; base += 4) {
        const int mt = min(4, cnt - base);
        const int mtb = mt <= 1 ? 1 : mt <= 2 ? 2 : 4;
        if (threadIdx.x < 8)
            tok[threadIdx.x] =
                threadIdx.x < mt ? list[base + threadIdx.x] / p.topk : -1;
        if (threadIdx.x == 0) s_mk = 0;
        __syncthreads();
        stage_x<BITS>(p.x, p.K, tok, mtb, p.nch, smem, &s_mk);
        __syncthreads();
        const bool mk = s_mk != 0;
        const int *l = list + base;
        if (mtb == 1)
            moe_gate_up_body<BITS, 1>(p, v, l, mt, i0, smem, mk);
        else if (mtb == 2)
            moe_gate_up_body<BITS, 2>(p, v, l, mt, i0, smem, mk);
        else
            moe_gate_up_body<BITS, 4>(p, v, l, mt, i0, smem, mk);
        __syncthreads();
    }
}

// ------------------------------------------------------------ down + combine
template <int BITS, int L, int D>
__global__ void __launch_bounds__(kMoeDownThreads)
    moe_down_kernel(MoeParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_tok[kMoeMaxSlots];
    __shared__ int s_first[kMoeMaxSlots];   // earliest slot with the same id
    __shared__ int s_gidx[kMoeMaxSlots];    // group index of a first slot
    __shared__ int s_gexp[kMoeMaxSlots];
    __shared__ int s_gstart[kMoeMaxSlots + 1];
    __shared__ int s_order[kMoeMaxSlots];
    __shared__ float s_rw[kMoeMaxSlots];
    __shared__ int s_ng;
    __shared__ int s_mk;  // some staged group is marked (common.cuh)
    const int S = p.M * p.topk;
    const int t = threadIdx.x;

    if (t == 0) s_mk = 0;
    // 1. earliest slot naming the same (valid) expert
    if (t < S) {
        const int e = p.ids[t];
        s_tok[t] = t;
        s_rw[t] = p.route_w[t];
        int f = -1;
        if (e >= 0 && e < p.E) {
            f = t;
            for (int s = 0; s < t; ++s)
                if (p.ids[s] == e) {
                    f = s;
                    break;
                }
        } else if (p.status && blockIdx.x == 0) {
            atomicOr(p.status, 1);
        }
        s_first[t] = f;
    }
    __syncthreads();
    // 2. groups in first-occurrence order, with their start offsets
    if (t < S && s_first[t] == t) {
        int gi = 0, start = 0;
        for (int s = 0; s < S; ++s) {
            gi += (s < t && s_first[s] == s);
            start += (s_first[s] >= 0 && s_first[s] < t);
        }
        s_gidx[t] = gi;
        s_gexp[gi] = p.ids[t];
        s_gstart[gi] = start;
    }
    if (t == 0) {
        int ng = 0, valid = 0;
        for (int s = 0; s < S; ++s) {
            ng += (s_first[s] == s);
            valid += (s_first[s] >= 0);
        }
        s_ng = ng;
        s_gstart[ng] = valid;
    }
    __syncthreads();
    // 3. slots of each group, in slot order
    if (t < S && s_first[t] >= 0) {
        const int f = s_first[t];
        int rank = 0;
        for (int s = f; s < t; ++s) rank += (s_first[s] == f);
        s_order[s_gstart[s_gidx[f]] + rank] = t;
    }
    stage_x<BITS>(p.x, p.K, s_tok, S, p.nch, smem, &s_mk);
    __syncthreads();
    const bool mk = s_mk != 0;

    const int lane = t & 31, warp = t >> 5;
    const int lg = lane / L, sub = lane % L;
    const int64_t row =
        (int64_t)blockIdx.x * (kMoeDownThreads / L) + warp * (32 / L) + lg;
    const int64_t rows[1] = {row < p.N ? row : -1};
    const int cpl = (p.nch + L - 1) / L;
    const int nitems = s_ng * cpl;
    const float2 *aux = x_aux<BITS>(smem, S, p.nch);

    float acc[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m] = 0.f;

    auto load = [&](int it, ChunkRegs<1> &cr, int &c) {
        const int gi = it / cpl;
        c = sub + (it - gi * cpl) * L;
        const int64_t e = s_gexp[gi];
        const WView v{reinterpret_cast<const uint4 *>(p.wq) + e * p.N * p.nch,
                      p.sc + e * p.N * p.G, p.bi + e * p.N * p.G, p.nch, p.G};
        if (c < p.nch) {
            load_chunk<BITS, 1>(v, rows, c, cr);
        } else {
            cr.w[0] = make_uint4(0, 0, 0, 0);
            cr.s[0] = cr.b[0] = 0.f;
        }
    };
    ChunkRegs<1> ring[D];
    int ringc[D];
#pragma unroll
    for (int k = 0; k < D; ++k)
        if (k < nitems) load(k, ring[k], ringc[k]);
    for (int base = 0; base < nitems; base += D) {
#pragma unroll
        for (int k = 0; k < D; ++k) {
            const int it = base + k;
            if (it >= nitems) break;
            const int c = ringc[k];
            if (c < p.nch) {
                const int gi = it / cpl;
                for (int q = s_gstart[gi]; q < s_gstart[gi + 1]; ++q) {
                    const int s = s_order[q];
                    const int midx[1] = {s};
                    float part[1][1] = {{0.f}};
                    if (mk)
                        chunk_fma<BITS, 1, 1, true>(ring[k], c, p.nch, midx, aux,
                                                    smem, part);
                    else
                        chunk_fma<BITS, 1, 1, false>(ring[k], c, p.nch, midx, aux,
                                                     smem, part);
                    const int tk = s / p.topk;
                    const float v = s_rw[s] * part[0][0];
#pragma unroll
                    for (int m = 0; m < 8; ++m) acc[m] += (m == tk) ? v : 0.f;
                }
            }
            if (it + D < nitems) load(it + D, ring[k], ringc[k]);
        }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m] = group_sum<L>(acc[m]);
    if (sub == 0 && row < p.N) {
#pragma unroll
        for (int m = 0; m < 8; ++m)
            if (m < p.M) p.out[(int64_t)m * p.N + row] = f32_to_bf16_bits(acc[m]);
    }
}

// ------------------------------------------------------------ host side
template <int BITS>
static size_t gate_up_stage_bytes(int nch) {
    return XStage<BITS>::bytes(4, nch);
}

template <int BITS>
static size_t down_stage_bytes(int S, int nch) {
    return XStage<BITS>::bytes(S, nch);
}

int moe_max_tokens(int bits, int nch, int mode) {
    // largest slot count (down) / token bucket (gate+up) whose staging fits
    if (mode == 0) {
        const size_t b = bits == 4 ? gate_up_stage_bytes<4>(nch)
                                   : gate_up_stage_bytes<8>(nch);
        return b <= kMaxDynSmem ? kMoeMaxSlots : 0;
    }
    int S = kMoeMaxSlots;
    while (S > 0 && (bits == 4 ? down_stage_bytes<4>(S, nch)
                               : down_stage_bytes<8>(S, nch)) > kMaxDynSmem)
        --S;
    return S;
}

template <int BITS>
static cudaError_t launch_gu(const MoeParams &p, cudaStream_t st) {
    auto kern = moe_gate_up_kernel<BITS>;
    const size_t smem = gate_up_stage_bytes<BITS>(p.nch);
    int dummy;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   kMoeThreads, smem, &dummy);
    if (e != cudaSuccess) return e;
    constexpr int kPairsPerCta = (kMoeThreads / 32) * kMoeRP;
    const int64_t I = p.N / 2;
    dim3 grid((unsigned)((I + kPairsPerCta - 1) / kPairsPerCta),
              (unsigned)(p.M * p.topk));
    kern<<<grid, kMoeThreads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_moe_gate_up(const MoeParams &p, cudaStream_t st) {
    return p.bits == 4 ? launch_gu<4>(p, st) : launch_gu<8>(p, st);
}

template <int BITS, int L>
static cudaError_t launch_dn(const MoeParams &p, cudaStream_t st) {
    auto kern = moe_down_kernel<BITS, L, 8>;
    const size_t smem = down_stage_bytes<BITS>(p.M * p.topk, p.nch);
    int dummy;
    cudaError_t e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   kMoeDownThreads, smem, &dummy);
    if (e != cudaSuccess) return e;
    constexpr int kRowsPerCta = kMoeDownThreads / L;
    const unsigned grid = (unsigned)((p.N + kRowsPerCta - 1) / kRowsPerCta);
    kern<<<grid, kMoeDownThreads, smem, st>>>(p);
    return cudaGetLastError();
}

template <int BITS>
static cudaError_t launch_dn_l(const MoeParams &p, cudaStream_t st) {
    if (p.nch >= 32) return launch_dn<BITS, 32>(p, st);
    if (p.nch >= 16) return launch_dn<BITS, 16>(p, st);
    return launch_dn<BITS, 8>(p, st);
}

cudaError_t launch_moe_down(const MoeParams &p, cudaStream_t st) {
    return p.bits == 4 ? launch_dn_l<4>(p, st) : launch_dn_l<8>(p, st);
}

}  // namespace gwa
