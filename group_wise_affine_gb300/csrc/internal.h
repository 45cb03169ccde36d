// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gwa {

// `bits` of fp8 (e4m3) weights (GWA_FP8_E4M3), and the stream width of a
// code of any format.
constexpr int kFp8 = 0x108;
__host__ __device__ constexpr int code_bits(int bits) {
    return bits == kFp8 ? 8 : bits;
}

constexpr int kDenseThreads = 512;
// Shared-memory budget (bytes) above which staged activations are kept as
// bf16 instead of fp32.
constexpr size_t kDenseF32StageMax = 96 * 1024;
// Dynamic shared memory the launchers budget per CTA: the sm_103a opt-in
// limit (227 KB) less room for the kernels' static arrays.
constexpr size_t kMaxDynSmem = 216 * 1024;
constexpr int kMaxSections = 8;
// Streaming decode kernel: largest CTA, and the shared-memory ring size it
// aims for per CTA.
constexpr int kStreamMaxThreads = 512;
constexpr size_t kStreamRingTarget = 96 * 1024;

struct DenseParams {
    const uint16_t *x;   // [M, K] bf16
    int M;               // tokens in this launch (<= 8)
    int K;
    int bits;
    const uint32_t *wq;  // [N, K*bits/32]
    const uint16_t *sc;  // [N, K/64]
    const uint16_t *bi;  // [N, K/64]
    int64_t N;           // weight rows
    int nch;             // 16-byte chunks per row
    int G;               // groups per row
    int group;           // inputs per group (the tuned kernels: 64)
    int64_t nblocks;     // warp blocks (set by the launcher)
    uint16_t *y;         // plain: [M, N]; gate+up: [M, I]
    int64_t I;           // gate+up: N / 2
    int nsec;
    int64_t sec_start[kMaxSections + 1];
    uint16_t *sec_out[kMaxSections];
    const uint16_t *sec_bias[kMaxSections];
    // rotary embedding (one-token kernel, QKV mode): rows [0, rope_end) are
    // rotated in heads of rope_hd at positions rope_pos[m]
    int rope_hd;
    int64_t rope_end;
    const int32_t *rope_pos;  // one-token kernel: forms its own (cos, sin)
    double rope_r;            // base^(-2/d), in fp64
    const float2 *rope_cs;    // staged kernel: (cos, sin) [M, rope_hd / 2]
};

// General-format decode kernel (qmv_generic.cu): u2/u4/u8 codes, groups of
// 32/64/128, up to generic_max_tokens() tokens per launch, modes as the
// other decode kernels (0 plain, 1 sections, 2 gate+up, 3 rotary sections).
cudaError_t launch_generic(int mode, const DenseParams &p, cudaStream_t st);
int generic_max_tokens();

// Attention over an affine-quantized value cache (attention.cu): partial
// softmax per key split into `part`, then the combine.
cudaError_t launch_attention(const uint16_t *q, const uint16_t *k,
                             const uint32_t *vq, const uint16_t *vs,
                             const uint16_t *vb, uint16_t *out, float *part,
                             int B, int Hq, int Hkv, int Lq, int T, int D,
                             int bits, float scale, int causal,
                             cudaStream_t st);
size_t attention_workspace_bytes(int B, int Hq, int Hkv, int Lq, int T, int D);

// (cos, sin) table of the rotary embedding, cs[m * d/2 + i] (rope.cu).
cudaError_t launch_rope_table(float2 *cs, int64_t M, int head_dim, double r,
                              const int32_t *positions, cudaStream_t st);

// Launches `kernel` on `st` with programmatic stream serialization: it may
// start while the previous kernel in the stream drains; the kernel itself
// waits (griddepcontrol.wait) before touching anything that kernel wrote.
template <typename... Args>
cudaError_t launch_pdl(const void *kernel, unsigned grid, unsigned threads,
                       size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *argv[] = {reinterpret_cast<void *>(&args)...};
    return cudaLaunchKernelExC(&cfg, kernel, argv);
}

// The same with thread-block clusters of `cluster` CTAs along x (grid a
// multiple of it).
template <typename... Args>
cudaError_t launch_pdl_cluster(const void *kernel, unsigned grid,
                               unsigned cluster, unsigned threads,
                               size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *argv[] = {reinterpret_cast<void *>(&args)...};
    return cudaLaunchKernelExC(&cfg, kernel, argv);
}

// Blocks for a persistent grid: SMs x resident CTAs of `kernel`.
cudaError_t occupancy_grid(const void *kernel, int threads, size_t smem,
                           int *grid);
int num_sms();
// Clusters of `cl` CTAs of `kernel` the GPU keeps resident at once (0: none;
// the kernel's shared-memory attribute set first, as occupancy_grid does).
int resident_clusters(const void *kernel, int cl, int threads, size_t smem);
// Largest shared-memory carveout for a streaming kernel (once per device).
cudaError_t prefer_max_shared(const void *kernel);

cudaError_t launch_dense(int mode, const DenseParams &p, cudaStream_t st);
cudaError_t launch_stream(int mode, const DenseParams &p, cudaStream_t st,
                          bool *used);
unsigned int stream_timeouts(bool reset);
// Tensor-core decode kernel, up to 8 tokens in one pass (qmv_mma.cu; used for
// 5..8 tokens); *used tells the caller whether the shape allowed it.
cudaError_t launch_mma(int mode, const DenseParams &p, cudaStream_t st,
                       bool *used);
unsigned int mma_timeouts(bool reset);
// One-token kernel with one quantization group per lane (qmv_group.cu).
// mode: 0 plain, 1 sections, 2 gate+up SiLU, 3 QKV sections with the
// rotary embedding of rows [0, p.rope_end)
cudaError_t launch_group(int mode, const DenseParams &p, cudaStream_t st,
                         bool *used);
unsigned int group_timeouts(bool reset);
// Whether the streaming kernel can run this shape (alignment, group count,
// row length); M is ignored.
bool stream_eligible(const DenseParams &p);
int dense_max_tokens(int bits, int nch);

struct MoeParams {
    const uint16_t *x;      // gate+up: [M, K]; down: [M, topk, K]
    int M;
    int topk;
    int K;
    int bits;
    const int32_t *ids;     // [M, topk]
    const float *route_w;   // [M, topk] (down)
    const uint32_t *wq;     // [E, N, K*bits/32]
    const uint16_t *sc;     // [E, N, K/64]
    const uint16_t *bi;
    int64_t N;              // rows per expert
    int E;
    int nch;
    int G;
    uint16_t *out;
    int32_t *status;
};
cudaError_t launch_moe_gate_up(const MoeParams &p, cudaStream_t st);
cudaError_t launch_moe_down(const MoeParams &p, cudaStream_t st);
int moe_max_tokens(int bits, int nch, int mode);
// Streaming MoE kernels (moe_stream.cu) for rows of up to 2048 inputs.
cudaError_t launch_moe_stream(int mode, const MoeParams &p, cudaStream_t st,
                              bool *used);
unsigned int moe_stream_timeouts(bool reset);

// Affine group quantization of bf16 weights (quantize.cu).
cudaError_t launch_quantize(const uint16_t *w, int64_t N, int64_t K, int bits,
                            uint32_t *wq, uint16_t *sc, uint16_t *bi,
                            cudaStream_t st);

cudaError_t launch_debug_unpack(const uint32_t *wq, int64_t N, int64_t K,
                                int bits, uint8_t *codes, cudaStream_t st);
cudaError_t launch_debug_dequant(const uint32_t *wq, const uint16_t *sc,
                                 const uint16_t *bi, int64_t N, int64_t K,
                                 int bits, int group, float *wf,
                                 cudaStream_t st);
cudaError_t launch_debug_wait(uint32_t *out, unsigned long long limit_ns,
                              cudaStream_t st);

}  // namespace gwa
