// Streaming top-k MoE expert GEMV ("Sanctum-MLX": 3-D switch_mlp expert
// grids; "Four Candles For The Cathedral", "What's not in this batch":
// routed experts with per-expert gate_proj / up_proj, and the 6x regression
// that came from duplicating expert weights).  Every distinct expert of the
// call is read once, in place, from the caller's stacked tensor.
//
// Same pipeline as the one-token decode kernel (qmv_group.cu): a producer
// thread fills a shared-memory ring
// with packed expert rows and their scales and biases by bulk copy, and
// consumer lanes each own one group of 64 inputs and form exact integer dots
// (group_dot.cuh).  A row's groups fit in one slice of W lanes (W = 8, 16 or
// 32 >= K/64), so a slice reduction yields the full row dot.  Scales and
// biases travel in the same stage as the codes: a pass then waits on shared
// memory only, where reading them from global memory a pass or two ahead
// left each short pass waiting a DRAM round trip.
//
// Routing.  Each CTA first groups the slots (token, k) by expert, in
// first-occurrence order, slots in slot order within a group.  Expert ids,
// route weights and weights are inputs no kernel of this library writes, and
// a kernel of any other kind completes before one of ours starts, so the
// grouping and the weight prefetch run before the wait on the previous
// kernel; only the activations (x, or the gate+up output h) wait for it.
//
// Gate+up mode.  Work units are (expert group, gate/up row pair); a CTA takes
// an even share of the units, and a stage holds up to UPS pairs of one
// expert (two copies: the gate rows and the up rows).  For every slot of the
// stage's expert the consumers form the gate and up dots of its token and
// write h[slot, i] = SiLU(g) * u.
//
// Down mode.  Clusters of CL CTAs (CL = 1, 2 or 4, as many as the GPU keeps
// resident in one wave): a cluster owns a block of output rows, and its CTA
// of rank c streams that block of the expert groups c, c + CL, ... (one copy
// per expert), adding route_w[slot] *
// (W[e] h[slot]) into its own accumulator of the slot's token.  At the end
// the CTAs of the cluster add the accumulators of ranks 0, 1, ... through
// distributed shared memory, so the combine is deterministic and needs no
// atomics or global scratch.

#include "cluster.cuh"
#include "group_dot.cuh"
#include "internal.h"

namespace gwa {

static __device__ unsigned int g_moe_timeouts;

// Eight warps at up to 128 registers: two CTAs (this kernel and the next one
// in the stream) fit in an SM's 64K registers.
constexpr int kMsConsumerWarps = 7;
constexpr int kMsThreads = (kMsConsumerWarps + 1) * kWarp;
// Dynamic shared memory per CTA: two CTAs per SM (228 KB, 1 KB reserved
// each) less the static routing tables.
constexpr size_t kMsSmemCap = 100 * 1024;
constexpr int kMsMaxSlots = 256;
constexpr int kMsMaxStages = 16;
constexpr int kMsMaxCluster = 8;    // down: CTAs sharing a row block
constexpr int kMsMaxRows = 128;     // down: output rows per cluster
constexpr size_t kMsStageTarget = 32 * 1024;

struct MsTables {
    int ids[kMsMaxSlots];
    int first[kMsMaxSlots];      // earliest slot with the same valid id, or -1
    int gidx[kMsMaxSlots];       // group of a first slot
    int gexp[kMsMaxSlots];       // expert of a group
    int gstart[kMsMaxSlots + 1]; // slot range of a group in `order`
    int order[kMsMaxSlots];      // slots grouped by expert
    int2 slotrow[kMsMaxSlots];   // order[q] and the image row of that slot
    int imgrow[kMsMaxSlots];     // image row holding a slot's activations
    int imgsrc[kMsMaxSlots];     // down: slot (source row) of an image row
    float rw[kMsMaxSlots];
    int ng, nimg;
};

// Stage k of this CTA: expert group, first unit, unit count.  Gate+up units
// are pairs of group gi; down units are output rows of the cluster's block.
struct MsStage {
    int gi, u, n;
};

// A CTA's stages in order; producer and consumers walk the same sequence
// (incremental, no division per stage).  Gate+up: units [u0, u1) of ng*I,
// cut at group ends.  Down: groups g0, g0 + step, ..., each the row block
// [u0, u1) in chunks of ups rows.
struct MsWalk {
    int mode, ups;
    int gi, ia, I;       // gate+up: group and unit within it
    int64_t cur, u1;     // gate+up: next unit, end
    int j, c, mine;      // down: group index among this rank's, chunk
    int g0, step, nchunk, r0, r1;
    __device__ void init_gate_up(int ups_, int64_t u0_, int64_t u1_, int I_) {
        mode = 0;
        ups = ups_;
        I = I_;
        cur = u0_;
        u1 = u1_;
        gi = (int)(u0_ / I_);
        ia = (int)(u0_ - (int64_t)gi * I_);
    }
    __device__ void init_down(int ups_, int ng, int g0_, int step_, int r0_,
                              int r1_) {
        mode = 1;
        ups = ups_;
        g0 = g0_;
        step = step_;
        r0 = r0_;
        r1 = r1_;
        nchunk = r1_ > r0_ ? (r1_ - r0_ + ups_ - 1) / ups_ : 0;
        mine = ng > g0_ && nchunk > 0 ? (ng - g0_ + step_ - 1) / step_ : 0;
        j = 0;
        c = 0;
    }
    __device__ bool next(MsStage &s) {
        if (mode == 0) {
            if (cur >= u1) return false;
            const int n = (int)min((int64_t)min(ups, I - ia), u1 - cur);
            s.gi = gi;
            s.u = ia;
            s.n = n;
            cur += n;
            ia += n;
            if (ia == I) {
                ++gi;
                ia = 0;
            }
            return true;
        }
        if (j >= mine) return false;
        s.gi = g0 + j * step;
        s.u = r0 + c * ups;
        s.n = min(ups, r1 - s.u);
        if (++c == nchunk) {
            c = 0;
            ++j;
        }
        return true;
    }
};

// One pass of the consumers over a stage: rows [sb, sb + sbu) of each half.
struct MsTask {
    MsStage sg;
    int k, sb;
    bool last;  // the stage's final pass
};

struct MsTasks {
    MsWalk w;
    MsStage sg;
    int k, sb, sbu;
    bool have;
    __device__ void init(const MsWalk &w0, int sbu_) {
        w = w0;
        sbu = sbu_;
        k = 0;
        sb = 0;
        have = w.next(sg);
    }
    __device__ bool next(MsTask &t) {
        if (!have) return false;
        t.sg = sg;
        t.k = k;
        t.sb = sb;
        t.last = sb + sbu >= sg.n;
        sb += sbu;
        if (sb >= sg.n) {
            sb = 0;
            ++k;
            have = w.next(sg);
        }
        return true;
    }
};

template <int BITS, int MODE, int W>
__global__ void __maxnreg__(128)
    moe_stream_kernel(MoeParams p, int stages, int rs, int ups, int cl,
                      uint32_t img_off, uint32_t acc_off) {
    constexpr int HALVES = MODE == 0 ? 2 : 1;
    // units per row group and pass (gate+up: row pairs, down: rows): two,
    // half the passes of one; more do not fit in the registers
    constexpr int UPT = 2;
    constexpr int RPH = HALVES * UPT;       // rows per lane and pass
    constexpr int GB = BITS * 8;            // code bytes per row and group
    const int CL = MODE == 0 ? 1 : cl;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ MsTables tb;
    __shared__ int s_issued, s_consumed;
    __shared__ int s_marked;  // some image group is marked (group_dot.cuh)
    // down: accumulators [row of the cluster block][token]
    float *acc = reinterpret_cast<float *>(smem + acc_off);

    const int tid = threadIdx.x;
    const int ncons = kMsConsumerWarps * kWarp;
    const int lane = tid & (kWarp - 1);
    const int S = p.M * p.topk;
    const int64_t I = p.N / 2;
    const int sbu = rs * UPT;
    const uint32_t rowbytes = (uint32_t)p.K * BITS / 8;
    const uint32_t sbrow = (uint32_t)p.G * 2;  // scale (bias) bytes per row
    // a stage: codes [half][ups rows], then scales, then biases, same order
    const uint32_t sc_off = (uint32_t)(HALVES * ups) * rowbytes;
    const uint32_t bi_off = sc_off + (uint32_t)(HALVES * ups) * sbrow;
    const uint32_t stage_bytes = bi_off + (uint32_t)(HALVES * ups) * sbrow;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    uint64_t *empty = full + stages;
    const int rank = CL > 1 ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    const int64_t blk0 = MODE == 1 ? p.N * cid / ncl : 0;
    const int64_t blk1 = MODE == 1 ? p.N * (cid + 1) / ncl : 0;
    const int nblk = (int)(blk1 - blk0);

    // ---------------------------------------------------- routing tables
    for (int s = tid; s < S; s += blockDim.x) {
        tb.ids[s] = p.ids[s];
        tb.rw[s] = MODE == 1 ? p.route_w[s] : 0.f;
    }
    if (MODE == 1)
        for (int i = tid; i < nblk * p.M; i += blockDim.x) acc[i] = 0.f;
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kMsConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    for (int s = tid; s < S; s += blockDim.x) {
        const int e = tb.ids[s];
        int f = -1;
        if (e >= 0 && e < p.E) {
            f = s;
            for (int q = 0; q < s; ++q)
                if (tb.ids[q] == e) {
                    f = q;
                    break;
                }
        } else if (p.status && blockIdx.x == 0) {
            atomicOr(p.status, 1);
        }
        tb.first[s] = f;
    }
    __syncthreads();
    for (int s = tid; s < S; s += blockDim.x) {
        if (tb.first[s] != s) continue;
        int gi = 0, start = 0;
        for (int q = 0; q < S; ++q) {
            gi += (q < s && tb.first[q] == q);
            start += (tb.first[q] >= 0 && tb.first[q] < s);
        }
        tb.gidx[s] = gi;
        tb.gexp[gi] = tb.ids[s];
        tb.gstart[gi] = start;
    }
    if (tid == 0) {
        int ng = 0, valid = 0;
        for (int q = 0; q < S; ++q) {
            ng += (tb.first[q] == q);
            valid += (tb.first[q] >= 0);
        }
        tb.ng = ng;
        tb.gstart[ng] = valid;
        s_issued = 0;
        s_consumed = 1 << 30;
        s_marked = 0;
    }
    __syncthreads();
    for (int s = tid; s < S; s += blockDim.x) {
        const int f = tb.first[s];
        if (f < 0) continue;
        int rank_in = 0;
        for (int q = f; q < s; ++q) rank_in += (tb.first[q] == f);
        tb.order[tb.gstart[tb.gidx[f]] + rank_in] = s;
    }
    __syncthreads();
    // image rows: gate+up, the tokens; down, this CTA's slots in group order
    if (tid == 0) {
        if (MODE == 0) {
            for (int s = 0; s < S; ++s) tb.imgrow[s] = s / p.topk;
            tb.nimg = p.M;
        } else {
            int n = 0;
            for (int gi = rank; gi < tb.ng; gi += CL)
                for (int q = tb.gstart[gi]; q < tb.gstart[gi + 1]; ++q) {
                    tb.imgrow[tb.order[q]] = n;
                    tb.imgsrc[n++] = tb.order[q];
                }
            tb.nimg = n;
        }
        pdl_launch_dependents();
    }
    __syncthreads();
    for (int q = tid; q < tb.gstart[tb.ng]; q += blockDim.x) {
        const int slot = tb.order[q];
        tb.slotrow[q] = make_int2(slot, tb.imgrow[slot]);
    }
    __syncthreads();

    // this CTA's stages
    MsWalk walk{};
    if (MODE == 0) {
        const int64_t units = (int64_t)tb.ng * I;
        walk.init_gate_up(ups, units * blockIdx.x / gridDim.x,
                          units * (blockIdx.x + 1) / gridDim.x, (int)I);
    } else {
        walk.init_down(ups, tb.ng, rank, CL, (int)blk0, (int)blk1);
    }

    if (tid >= ncons) {
        // ------------------------------------------------ producer
        if (tid == ncons) {
            const unsigned char *wq =
                reinterpret_cast<const unsigned char *>(p.wq);
            const unsigned char *sc =
                reinterpret_cast<const unsigned char *>(p.sc);
            const unsigned char *bi =
                reinterpret_cast<const unsigned char *>(p.bi);
            MsWalk w = walk;
            MsStage sg;
            int k = 0, s = 0;
            uint32_t ph = 0;  // use count parity of slot s
            while (w.next(sg)) {
                if (k >= stages && !mbar_wait(&empty[s], ph ^ 1)) {
                    atomicAdd(&g_moe_timeouts, 1u);
                    break;
                }
                const int64_t e = tb.gexp[sg.gi];
                unsigned char *base = smem + (size_t)s * stage_bytes;
                mbar_expect_tx(&full[s], (uint32_t)(HALVES * sg.n) *
                                             (rowbytes + 2 * sbrow));
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                    const int64_t r = e * p.N + sg.u + (h ? I : 0);
                    bulk_g2s(base + (size_t)h * ups * rowbytes,
                             wq + r * rowbytes, sg.n * rowbytes, &full[s]);
                    bulk_g2s(base + sc_off + (size_t)h * ups * sbrow,
                             sc + r * sbrow, sg.n * sbrow, &full[s]);
                    bulk_g2s(base + bi_off + (size_t)h * ups * sbrow,
                             bi + r * sbrow, sg.n * sbrow, &full[s]);
                }
                s_issued = ++k;
                if (++s == stages) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
    } else {
        // ------------------------------------------------ consumers
        const int hg = tid / W;                 // row group
        const bool in_group = hg < rs;
        const int hgc = in_group ? hg : 0;
        const int g = tid & (W - 1);
        const bool active = in_group && g < p.G;
        const int gg = active ? g : 0;
        const int rot = chunk_rot<BITS>(gg);
        unsigned char *img = smem + img_off;

        MsTasks tasks;
        tasks.init(walk, sbu);

        pdl_wait_primary();  // x / h may be the previous kernel's output
        encode_rows_shared<BITS>(p.x, tb.nimg, tb.nimg, p.K, p.G, tid, ncons,
                                 img, MODE == 1 ? tb.imgsrc : nullptr, &s_marked);
        asm volatile("bar.sync 1, %0;" ::"r"(ncons) : "memory");
        const bool img_marked = s_marked != 0;

        GroupX<1> gx;
        int cached = -1;
        int s = -1;       // ring slot of the current stage
        uint32_t ph = 1;  // its use count parity
        // The task loop, once with the marked-group path (EX) and once
        // without it (see qmv_group.cu); the image rows a lane reads change
        // over the loop, so the choice is made from every row of the image.
        auto task_loop = [&](auto ex) {
            constexpr bool EX = decltype(ex)::value;
            MsTask t;
            while (tasks.next(t)) {
                if (t.sb == 0) {
                    if (++s == stages) s = 0;
                    if (s == 0) ph ^= 1;
                    if (!mbar_wait(&full[s], ph)) {
                        atomicAdd(&g_moe_timeouts, 1u);
                        atomicMin(&s_consumed, t.k);
                        break;
                    }
                }
                const unsigned char *base = smem + (size_t)s * stage_bytes;
                const int pos = t.sb + hgc * UPT;
                const int q1 = tb.gstart[t.sg.gi + 1];
                for (int qi = tb.gstart[t.sg.gi]; qi < q1; ++qi) {
                    const int2 sr = tb.slotrow[qi];
                    const int slot = sr.x, row = sr.y;
                    if (row != cached) {
                        load_group_rows<1>(img, tb.nimg, p.G, row, gg, active, gx,
                                           image_shift<BITS>(gg));
                        cached = row;
                    }
                    float v[RPH];
#pragma unroll
                    for (int j = 0; j < RPH; ++j) {
                        // stage row of value j (rows past the stage's end read
                        // its last row, finite, and are not stored)
                        const uint32_t roj = (uint32_t)((j / UPT) * ups +
                                                        min(pos + (j % UPT), t.sg.n - 1));
                        uint4 wv[BITS / 2];
                        lds_group<BITS>(base + roj * rowbytes + (uint32_t)gg * GB,
                                        rot, wv);
                        const uint32_t so = (roj * (uint32_t)p.G + gg) * 2u;
                        const float sv = bf16_bits_to_f32(
                            *reinterpret_cast<const uint16_t *>(base + sc_off + so));
                        const float bv = bf16_bits_to_f32(
                            *reinterpret_cast<const uint16_t *>(base + bi_off + so));
                        int d[1];
                        group_dot<BITS, 1>(wv, gx, d);
                        float df = (float)d[0];
                        if (EX && gx.mk[0])  // marked group: fp32 dot of raw x
                            df = group_dot_f32<BITS, 1>(wv, gx, 0);
                        v[j] = fmaf(sv * gx.f[0], df, bv * gx.xs[0]);
                        // keep the next row's loads after this dot (registers)
                        asm volatile("" ::: "memory");
                    }
                    // value j ends in slice lane j * (W / RPH); the second half's
                    // values (up rows, or down's odd rows) sit W/2 lanes up
                    const float tot = sub_reduce<W, RPH>(v, lane);
                    const float tot1 = __shfl_down_sync(0xffffffffu, tot, W / 2);
                    constexpr int SPREAD = W / RPH;
                    const int j = g / SPREAD;  // value index of this lane
                    if (in_group && g % SPREAD == 0 && g < W / 2) {
                        if (MODE == 0) {
                            // pair pos + j: gate value j, up value UPT + j
                            if (pos + j < t.sg.n)
                                p.out[(int64_t)slot * I + t.sg.u + pos + j] =
                                    f32_to_bf16_bits(tot / (1.0f + __expf(-tot)) *
                                                     tot1);
                        } else if (j == 0 && pos < t.sg.n) {
                            // rows pos (value 0) and pos + 1 (value 1)
                            const int tk = slot / p.topk;
                            const float r = tb.rw[slot];
                            float *a = acc + (size_t)(t.sg.u - blk0 + pos) * p.M + tk;
                            a[0] += r * tot;
                            if (pos + 1 < t.sg.n) a[p.M] += r * tot1;
                        }
                    }
                }
                if (t.last) {
                    // every lane's reads of this stage are done: release it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
            }
        };
        if (img_marked)
            task_loop(std::true_type{});
        else
            task_loop(std::false_type{});
    }
    __syncthreads();
    // Outputs are written by consumer threads only: they passed the
    // dependency wait before reading the activations, so the previous grid
    // (which may read what the outputs alias) is complete.
    // A timed-out pipeline must not leave bulk copies landing in shared
    // memory after the CTA exits: wait (again bounded) for every stage that
    // was issued but not consumed.
    if (tid == ncons && s_consumed < s_issued) {
        for (int k = s_consumed; k < s_issued; ++k)
            if (!mbar_wait(&full[k % stages], (k / stages) & 1)) break;
    }

    if (MODE == 0) {
        // slots with an invalid expert: zero outputs, split over the CTAs
        const int64_t i0 = I * blockIdx.x / gridDim.x;
        const int64_t i1 = I * (blockIdx.x + 1) / gridDim.x;
        for (int s = 0; s < S && tid < ncons; ++s) {
            if (tb.first[s] >= 0) continue;
            for (int64_t i = i0 + tid; i < i1; i += ncons)
                p.out[(int64_t)s * I + i] = 0;
        }
    } else {
        // every CTA of the cluster has finished its accumulators; rank c
        // writes its share of the block, adding the ranks in order
        cluster_sync_all();
        const int r0 = nblk * rank / CL, r1 = nblk * (rank + 1) / CL;
        for (int i = tid; i < (r1 - r0) * p.M && tid < ncons; i += ncons) {
            const int r = r0 + i / p.M, t = i % p.M;
            // all ranks' loads in flight at once, then added in rank order
            float part[kMsMaxCluster];
#pragma unroll
            for (int q = 0; q < kMsMaxCluster; ++q)
                part[q] = q < CL ? ld_cluster_f32(acc + (size_t)r * p.M + t,
                                                  (uint32_t)q)
                                 : 0.f;
            float y = 0.f;
#pragma unroll
            for (int q = 0; q < kMsMaxCluster; ++q)
                if (q < CL) y += part[q];
            p.out[(int64_t)t * p.N + blk0 + r] = f32_to_bf16_bits(y);
        }
        // no CTA leaves while another still reads its accumulators
        cluster_sync_all();
    }
}

// ------------------------------------------------------------ host side

template <int BITS, int MODE, int W>
static cudaError_t launch_ms(const MoeParams &p, cudaStream_t st, bool *used) {
    constexpr int HALVES = MODE == 0 ? 2 : 1;
    constexpr int UPT = 2;
    const int S = p.M * p.topk;
    const size_t rowbytes = (size_t)p.K * BITS / 8;
    const size_t sbrow = (size_t)p.G * 2;
    const int rs = kMsConsumerWarps * kWarp / W;  // row groups per pass
    const int sbu = rs * UPT;
    int grid, ups, img_rows, nblk = 0, cl = 1;
    if (MODE == 0) {
        grid = num_sms();
        // a stage holds whole passes, about kMsStageTarget bytes, and no
        // more than a CTA's share
        int passes = (int)(kMsStageTarget /
                           ((size_t)HALVES * (rowbytes + 2 * sbrow) * sbu));
        if (passes < 1) passes = 1;
        ups = passes * sbu;
        const int64_t share = ((int64_t)S * (p.N / 2) + grid - 1) / grid;
        if ((int64_t)ups > share) ups = (int)(share > 0 ? share : 1);
        img_rows = p.M;
    } else {
        img_rows = S;
    }
    auto kern = moe_stream_kernel<BITS, MODE, W>;
    const size_t img = ximg_bytes(img_rows, p.G);
    size_t stage_bytes = 0, accb = 0, img_off = 0, acc_off = 0, smem = 0;
    int stages = 0;
    cudaError_t e;
    // shared-memory layout for a stage of `ups` units; false if the ring
    // gets fewer than two stages (or a down block exceeds kMsMaxRows)
    auto layout = [&]() -> bool {
        stage_bytes = (size_t)HALVES * ups * (rowbytes + 2 * sbrow);
        accb = MODE == 1 ? (size_t)nblk * p.M * 4 : 0;
        const size_t fixed = 16 * kMsMaxStages + ((img + 15) / 16) * 16 + accb;
        if (fixed >= kMsSmemCap) return false;
        stages = (int)((kMsSmemCap - fixed) / stage_bytes);
        if (stages > kMsMaxStages) stages = kMsMaxStages;
        img_off = stages * stage_bytes + 16 * stages;
        acc_off = img_off + ((img + 15) / 16) * 16;
        smem = acc_off + accb;
        return stages >= 2 && (MODE == 0 || nblk <= kMsMaxRows);
    };
    if (MODE == 0) {
        if (!layout()) return cudaSuccess;  // not used
        int dummy = 0;
        e = occupancy_grid(reinterpret_cast<const void *>(kern), kMsThreads,
                           smem, &dummy);
        if (e != cudaSuccess) return e;
    } else {
        // Clusters of up to kMsMaxCluster CTAs, one CTA per SM: the largest
        // size of which one wave keeps at least 90% of the SMs busy.  Only
        // the clusters one wave holds are launched (a GPC whose SM count
        // the size does not divide leaves a few SMs out).
        bool ok = false;
        for (cl = kMsMaxCluster; cl >= 1 && !ok; cl /= 2) {
            int clusters = num_sms() / cl;
            if ((int64_t)clusters > p.N) clusters = (int)p.N;
            for (int round = 0; round < 2 && !ok; ++round) {
                nblk = (int)((p.N + clusters - 1) / clusters);
                ups = (nblk + UPT - 1) / UPT * UPT;  // one stage per expert
                if (!layout()) break;
                int dummy = 0;
                e = occupancy_grid(reinterpret_cast<const void *>(kern),
                                   kMsThreads, smem, &dummy);
                if (e != cudaSuccess) return e;
                const int res =
                    cl == 1 ? clusters
                            : resident_clusters(
                                  reinterpret_cast<const void *>(kern), cl,
                                  kMsThreads, smem);
                if (res >= clusters) {
                    ok = true;
                    grid = clusters * cl;
                    break;
                }
                // longer blocks over fewer clusters, if enough SMs stay busy
                if ((int64_t)res * cl * 10 < (int64_t)num_sms() * 9) break;
                clusters = res;
            }
            if (ok) break;
        }
        if (!ok) return cudaSuccess;  // not used
    }
    e = prefer_max_shared(reinterpret_cast<const void *>(kern));
    if (e != cudaSuccess) return e;
    *used = true;
    if (MODE == 0)
        return launch_pdl(reinterpret_cast<const void *>(kern), grid,
                          kMsThreads, smem, st, p, stages, rs, ups, 1,
                          (uint32_t)img_off, (uint32_t)acc_off);
    return launch_pdl_cluster(reinterpret_cast<const void *>(kern), grid,
                              (unsigned)cl, kMsThreads, smem, st, p, stages,
                              rs, ups, cl, (uint32_t)img_off,
                              (uint32_t)acc_off);
}

template <int BITS, int MODE>
static cudaError_t launch_ms_w(const MoeParams &p, cudaStream_t st,
                               bool *used) {
    if (p.G <= 8) return launch_ms<BITS, MODE, 8>(p, st, used);
    if (p.G <= 16) return launch_ms<BITS, MODE, 16>(p, st, used);
    return launch_ms<BITS, MODE, 32>(p, st, used);
}

// Launches the streaming MoE kernel when the shape allows it (K <= 2048 and
// a multiple of 512, 16-byte aligned codes, scales, biases and activations,
// the encoded activations within the
// shared-memory budget); *used tells the caller whether it ran.
cudaError_t launch_moe_stream(int mode, const MoeParams &p, cudaStream_t st,
                              bool *used) {
    *used = false;
    auto a16 = [](const void *q) {
        return (reinterpret_cast<uintptr_t>(q) & 15) == 0;
    };
    if (p.G > 32 || (p.G % 8) != 0 || !a16(p.wq) || !a16(p.sc) ||
        !a16(p.bi) || !a16(p.x) || p.M * p.topk > kMsMaxSlots ||
        p.N >= (int64_t)1 << 30)
        return cudaSuccess;
    if (mode == 0)
        return p.bits == 4 ? launch_ms_w<4, 0>(p, st, used)
                           : launch_ms_w<8, 0>(p, st, used);
    return p.bits == 4 ? launch_ms_w<4, 1>(p, st, used)
                       : launch_ms_w<8, 1>(p, st, used);
}

unsigned int moe_stream_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_moe_timeouts, sizeof v);
    if (reset) {
        const unsigned int z = 0;
        cudaMemcpyToSymbol(g_moe_timeouts, &z, sizeof z);
    }
    return v;
}

}  // namespace gwa
