/*
 * gwa.h -- C ABI of libgwa.so: affine group-quantized linear projections on
 * one NVIDIA GB300 (sm_103a).
 *
 * The operation (MLX-style affine integer weights):
 *   code   q[n,k] = bits [b*k, b*k + b) of row n's little-endian bit stream
 *          (word j holds stream bits [32j, 32j + 32)); for b dividing 32
 *          that is (Wq[n, k/P] >> (b*(k mod P))) & (2^b - 1),  P = 32/b
 *   weight w[n,k] = scale[n, k/64] * q[n,k] + bias[n, k/64]
 *   output y[m,n] = sum_k x[m,k] * w[n,k]   (fp32 accumulation, bf16 out)
 * Defined by: "Sanctum-MLX", server diagram and model parameter table
 * (4-bit QuantizedLinear, group_size=64); "saragossa", "Quantization
 * formats" (MLX affine u2/u3/u4/u6/u8, group size 64, bf16 scales/biases,
 * u3 ~3.5, u4 ~4.5, u6 ~6.5, u8 ~8.5 bits per weight); "The Cathedral Doubled Itself", "The two fusions"
 * (packed weight [rows, hidden/8] uint32 for 4-bit codes, codes packed along
 * the input axis).  Inside a word the first code sits in the lowest bits.
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; arrays of
 *     pointers (section outputs/biases) and section sizes are HOST arrays.
 *     The library allocates nothing, keeps no pointer after the call returns,
 *     and never synchronizes: work is enqueued on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream) and the call returns at once.  (One
 *     exception: gwa_qmv_affine_noalloc runs in a fixed scratch buffer that
 *     the library holds in device memory for the life of the process.)
 *   - bf16 values are passed as their 16-bit patterns (uint16_t).
 *   - All matrices are row-major and contiguous.  x is [M, K].
 *   - Wq, x and the workspace must be 16-byte aligned; scales, biases and
 *     outputs 2-byte aligned.  K must be a multiple of 64.
 *   - bits is 2, 3, 4, 6 or 8; group 32, 64 or 128 (see gwa_qweight).
 *   - M <= 8 runs the decode (GEMV) kernels on the CUDA cores and needs no
 *     workspace (pass NULL, 0).  M > 8 needs `gwa_workspace_bytes(M, K)`
 *     bytes of device workspace, which the call overwrites; calls sharing one
 *     workspace must not overlap on the GPU.  It runs the tensor-core
 *     (tcgen05) kernels when K is a multiple of 512 and Wq, scales and
 *     biases are 16-byte aligned (the workspace's first word then holds the
 *     call's status: 0, or 1 when a pipeline wait ran out, which
 *     gwa_pipeline_status also counts), and otherwise the decode kernels in
 *     passes of up to 8 tokens.  Every finite bf16 input is in range: each
 *     token and each weight row is scaled by a power of two before the
 *     tensor cores' fp16 operands are formed.
 *   - Return value: GWA_OK or an error code; nothing aborts, traps or exits.
 *     On error nothing was enqueued and gwa_last_error() (thread-local) holds
 *     one line of text.  Errors raised by the GPU while the work runs surface
 *     from the next CUDA call that observes them, as usual for CUDA.
 */
#ifndef GWA_H_
#define GWA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    GWA_OK = 0,
    GWA_ERR_INVALID_ARG = 1, /* null pointer, bad size, sizes not adding up */
    GWA_ERR_UNSUPPORTED = 2, /* bits not in {2,3,4,6,8,GWA_FP8_E4M3}, group not in
                                {32,64,128}; or a format an entry point does
                                not take (experts, quantization: u4/u8 at
                                group 64)                                  */
    GWA_ERR_MISALIGNED = 3,  /* a pointer breaks the alignment rules       */
    GWA_ERR_CUDA = 4,        /* launch failed or no usable sm_103a device   */
    GWA_ERR_WORKSPACE = 5    /* M > 8 and the workspace is null or small    */
};

/* One packed weight of N output rows and K inputs (K a multiple of 64 and
 * of the group).
 *   wq:     uint32 [N, K*bits/32]: the row's codes along the input axis as
 *           one little-endian bit stream, lowest bits first (32/bits per
 *           word for u2/u4/u8; u3 and u6 codes may straddle two words)
 *   scales: bf16   [N, K/group]
 *   biases: bf16   [N, K/group]
 * bits 4 or 8 with group 64 run the tuned kernels; every other width and
 * group (u2, u3, u6 at any group; u4, u8 at 32 or 128) runs a general decode
 * kernel for the dense
 * projections (all of gwa_qmv_affine, gwa_qmv_fused_sections,
 * gwa_qmv_gate_up_silu, gwa_qmv_qkv_rope, the debug exports); the experts
 * and the quantization take u4/u8 at group 64 only.
 * bits = GWA_FP8_E4M3: 8-bit floating-point codes (OCP FP8 E4M3: 1 sign,
 * 4 exponent bits of bias 7, 3 mantissa bits, subnormals, no infinities,
 * S.1111.111 = NaN) packed four per word, lowest byte first, in the same
 * container: w = scale * e4m3(q) + bias ("saragossa", "Quantization
 * formats" lists fp8 (e4m3) beside the affine widths and gives it the u8
 * footprint, ~8.5 bits per weight).  Dense projections only, any group, on
 * the general decode kernel in fp32 (every product e4m3 * bf16 is exact). */
#define GWA_FP8_E4M3 0x108
typedef struct gwa_qweight {
    const uint32_t *wq;
    const uint16_t *scales;
    const uint16_t *biases;
    int64_t N;
    int64_t K;
    int32_t bits;
    int32_t group;
} gwa_qweight;

/* y[M, N] (bf16) = x[M, K] . dequant(w)^T.
 * The quantized linear layer itself ("Sanctum-MLX": QuantizedLinear
 * group_size=64; "The Cathedral Doubled Itself": quantized_matmul). */
int gwa_qmv_affine(const uint16_t *x, int64_t M, gwa_qweight w, uint16_t *y,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Fused projection over output-axis-concatenated weights, written back as
 * SEPARATE contiguous buffers.  ("The Cathedral Doubled Itself", "The two
 * fusions" and "The trap that ate three hours": one quantized_matmul over
 * [q_out + 2*kv_out, hidden/8], split on the last axis; split views with a
 * non-zero offset and the parent's strides corrupted RoPE, so every section
 * here is its own offset-0 row-major buffer.)
 *   w.N == sum(section_sizes[0 .. n_sections-1]); 1 <= n_sections <= 8.
 *   outs[s]:     device bf16 [M, section_sizes[s]], contiguous; rows
 *                [start_s, start_s + size_s) of the fused weight land there.
 *   out_bias:    NULL, or a host array of n_sections device pointers (each
 *                NULL or bf16 [section_sizes[s]]) added to that section's
 *                output in fp32 before rounding (the additive q/k/v bias of
 *                the qwen2 layout).
 * The buffers must not overlap each other or x. */
int gwa_qmv_fused_sections(const uint16_t *x, int64_t M, gwa_qweight w,
                           int32_t n_sections, const int64_t *section_sizes,
                           uint16_t *const *outs,
                           const uint16_t *const *out_bias, void *workspace,
                           size_t workspace_bytes, void *stream);

/* Fused gate+up projection with the SwiGLU epilogue.  ("The Cathedral
 * Doubled Itself", "The two fusions", Phase 1B: gate_proj and up_proj fused
 * the same way, ahead of SiLU and the multiply; no additive bias.)
 *   w has 2*I rows: rows [0, I) are gate_proj, rows [I, 2I) are up_proj.
 *   h[M, I] (bf16) = SiLU(g) * u with g, u the fp32 projections and
 *   SiLU(g) = g / (1 + exp(-g)), rounded to bf16 once. */
int gwa_qmv_gate_up_silu(const uint16_t *x, int64_t M, gwa_qweight w,
                         uint16_t *h, void *workspace, size_t workspace_bytes,
                         void *stream);

/* Workspace bytes the three dense entry points need for M tokens of K
 * inputs (0 when M <= 8). */
size_t gwa_workspace_bytes(int64_t M, int64_t K);

enum { GWA_MOE_GATE_UP_SILU = 0, GWA_MOE_DOWN_COMBINE = 1 };

/* Top-k MoE expert projection over stacked expert weights ("Sanctum-MLX":
 * 3-D switch_mlp expert grids; "Four Candles For The Cathedral", "What's not
 * in this batch": per-expert gate_proj/up_proj of the routed experts).
 *   w: stacked experts -- expert e owns rows [e*w.N, (e+1)*w.N) of wq,
 *      scales and biases, i.e. wq is [num_experts, w.N, K*bits/32].
 *   expert_ids: device int32 [M, topk].
 *   mode GWA_MOE_GATE_UP_SILU: x is [M, K]; each expert's w.N = 2*I rows are
 *      [gate; up]; out[M, topk, I] (bf16) = SiLU(Wg[e] x_t) * (Wu[e] x_t)
 *      for e = expert_ids[t, j].  route_w is ignored (may be NULL).
 *   mode GWA_MOE_DOWN_COMBINE: x is [M, topk, K] (one input per slot, e.g.
 *      the gate+up output); route_w is device fp32 [M, topk];
 *      out[M, w.N] (bf16) = sum_j route_w[t,j] * (W[e] x[t,j]), in fp32.
 *   Each distinct expert is streamed from memory once per call, however many
 *   tokens chose it.  1 <= M <= 8 and 1 <= topk <= 32.
 *   status: NULL, or a device int32 the kernels set to 1 (atomic OR) when an
 *      expert id lies outside [0, num_experts); such a slot contributes zero
 *      (gate+up mode writes zeros for it).  The caller clears it. */
int gwa_moe_qmv_gather(const uint16_t *x, int64_t M, int32_t topk,
                       const int32_t *expert_ids, const float *route_w,
                       gwa_qweight w, int32_t num_experts, int32_t mode,
                       uint16_t *out, int32_t *status, void *stream);

/* Allocation-free variant of gwa_qmv_affine, for callers that cannot
 * allocate device memory: for example a plug-in inside a host framework that
 * owns all device memory, or a serving loop that must not make allocation
 * calls (they can synchronize the device or fail under memory pressure in
 * the middle of a request).  Those callers cannot supply the workspace that
 * the tensor-core path (M > 8) needs, so this entry point uses a scratch
 * buffer of GWA_NOALLOC_SCRATCH_BYTES that the library itself holds in
 * device memory on every GPU that loads it, until the process exits.  It
 * allocates nothing and frees nothing.  (The pages have no counterpart:
 * this is a property of this library's interface, not of the method.)
 *   Same arguments, layout and results as gwa_qmv_affine, minus the
 *   workspace.  M <= 8 needs no scratch; for M > 8 the problem must fit:
 *   gwa_workspace_bytes(M, K) <= GWA_NOALLOC_SCRATCH_BYTES, otherwise the
 *   call returns GWA_ERR_WORKSPACE and enqueues nothing.
 *   Each call looks up the scratch's device address on the current device
 *   (cudaGetSymbolAddress) and keeps nothing between calls.
 *   Every call on a device shares the one scratch buffer and leaves its
 *   contents behind (the status word is cleared at the start of each call):
 *   calls that can overlap on the GPU -- on different streams, or from
 *   different host threads -- race on it and must be serialized by the
 *   caller.
 *   Status: the only condition the scratch's status word can record is a
 *   pipeline wait that ran out, and every such wait is also counted on the
 *   device, so gwa_pipeline_status reports it; the caller needs no access to
 *   the scratch.
 *   Size: gwa_workspace_bytes(M, K) is about 2.1 K bytes per token, so the
 *   scratch fits M <= 1925 at K = 2048, M <= 779 at K = 5120 and M <= 287
 *   at K = 13824 (a down projection); larger problems need gwa_qmv_affine
 *   with a workspace. */
#define GWA_NOALLOC_SCRATCH_BYTES (8u << 20)
int gwa_qmv_affine_noalloc(const uint16_t *x, int64_t M, gwa_qweight w,
                           uint16_t *y, void *stream);

/* gwa_qmv_qkv_rope -- the fused QKV projection (gwa_qmv_fused_sections with
 * the three sections Q, K, V) followed by the rotary position embedding of Q
 * and K: the step the pages design after the fused projection ("The
 * Cathedral Doubled Itself", "The kernel that worked and the kernel that
 * won't": RoPE on the materialized Q and K; "The trap that ate three hours":
 * RoPE runs per head at the cache offset).  The pages give no formula; this
 * library uses the textbook one with the rotate-half pairing: for every head
 * of head_dim = d in Q and in K, and i < d/2,
 *   t = positions[m] * rope_base^(-2i/d),
 *   (y[i], y[i + d/2]) -> (y[i] cos t - y[i + d/2] sin t,
 *                          y[i + d/2] cos t + y[i] sin t),
 * applied after the optional per-output bias; V is not rotated.  No frequency
 * scaling (YaRN and the like) is applied.
 *   w          fused weight, rows [0, q_size) = Q, then K, then V (kv_size
 *              each); q_size and kv_size multiples of head_dim.
 *   head_dim   even, 2..256.  rope_base > 0 (e.g. 10000 or 1e6).
 *   positions  int32 [M] on the device: the position of each token (cache
 *              offset + index); read as an input (no kernel of this library
 *              writes it).
 *   q, k, v    outputs [M, q_size], [M, kv_size], [M, kv_size], contiguous.
 *   out_bias   NULL or three bias pointers (each NULL or bf16 [size]).
 *   workspace  at least gwa_qkv_rope_workspace_bytes(M, K, head_dim)
 *              bytes, 256-byte aligned, for M > 1 (a (cos, sin) table, and
 *              for M > 8 the tensor-core path's area); M = 1 needs none when
 *              K is a multiple of 512 and the weight 16-byte aligned
 *              (otherwise as M > 1).  Its contents are scratch.
 * Every path rotates the fp32 projection before rounding to bf16.  One
 * token runs in one kernel (the rotation in the epilogue, its (cos, sin)
 * formed by the kernel); more tokens run a small kernel that fills the table
 * (angles in fp64, reduced modulo 2 pi), then the staged decode kernels (up
 * to eight tokens a pass) or, for M > 8 with head_dim dividing 128 and
 * q_size, kv_size multiples of 128, the tensor-core kernel, each rotating in
 * its epilogue.  Errors as gwa_qmv_fused_sections, plus
 * GWA_ERR_INVALID_ARG for head_dim, sizes, rope_base or a null positions
 * pointer, and GWA_ERR_WORKSPACE for a missing or short workspace. */
int gwa_qmv_qkv_rope(const uint16_t *x, int64_t M, gwa_qweight w,
                     int64_t q_size, int64_t kv_size, int32_t head_dim,
                     double rope_base, const int32_t *positions, uint16_t *q,
                     uint16_t *k, uint16_t *v,
                     const uint16_t *const *out_bias, void *workspace,
                     size_t workspace_bytes, void *stream);

/* Workspace bytes gwa_qmv_qkv_rope needs for M tokens of K inputs and
 * heads of head_dim (0 for M < 1). */
size_t gwa_qkv_rope_workspace_bytes(int64_t M, int64_t K, int32_t head_dim);

/* gwa_sdpa_dequant_v -- softmax attention over a quantized value cache,
 * the values dequantized inline ("Sanctum-MLX", six-changes table row 5,
 * "Fused attention with inline V dequant (sdpa_dequant_v)", and the
 * paragraph after it: Q, a materialized bf16 K and the compressed V state
 * in; fp32 online softmax; causal mask; GQA without copying K or V).  The
 * pages do not print the value format; this library's reading is its own
 * affine format along the head dimension: codes packed 32/bits per word,
 * lowest bits first, one bf16 scale and bias ("zero") per 64 dimensions,
 * v = scale * code + bias.
 *   out[b,h,l,:] = sum_t p_t v[b,h',t,:],  p = softmax_t(scale * q[b,h,l,:] .
 *   k[b,h',t,:]) over t < T (causal: t <= T - Lq + l, the queries being the
 *   last Lq positions), h' = h / (Hq / Hkv).
 *   q    bf16 [B, Hq, Lq, D];  k  bf16 [B, Hkv, T, D]   (16-byte aligned)
 *   vq   uint32 [B, Hkv, T, D*bits/32]                   (8-byte aligned)
 *   vs, vb  bf16 [B, Hkv, T, D/64]                       (8-byte aligned)
 *   out  bf16 [B, Hq, Lq, D]
 *   D 64, 128 or 256; bits 4 or 8; group 64; Hq a multiple of Hkv; T >= 1;
 *   causal needs Lq <= T.  scale is usually 1/sqrt(D).
 *   workspace  >= gwa_sdpa_workspace_bytes(...), 16-byte aligned (per-split
 *              partial softmax states).
 * Two kernels on `stream`: the keys of each (batch, KV head) split over the
 * GPU (scores and value products on the tensor cores, bf16 operands with
 * fp32 accumulation: the softmax weights times the value scales enter the
 * value product rounded to bf16), then a combine.  Errors: GWA_ERR_UNSUPPORTED (D, bits, group),
 * GWA_ERR_INVALID_ARG (shapes, null pointers, causal with Lq > T),
 * GWA_ERR_MISALIGNED, GWA_ERR_WORKSPACE; nothing is enqueued on error. */
int gwa_sdpa_dequant_v(const uint16_t *q, int64_t B, int32_t Hq, int32_t Lq,
                       int32_t D, const uint16_t *k, int32_t Hkv, int64_t T,
                       const uint32_t *vq, const uint16_t *vs,
                       const uint16_t *vb, int32_t bits, int32_t group,
                       float scale, int32_t causal, uint16_t *out,
                       void *workspace, size_t workspace_bytes, void *stream);
size_t gwa_sdpa_workspace_bytes(int64_t B, int32_t Hq, int32_t Hkv, int32_t Lq,
                                int64_t T, int32_t D);

/* gwa_quantize_affine -- affine group quantization of bf16 weights into the
 * packed format every projection above reads: the requantize step of
 * "Sanctum-MLX", "The April 2026 cutover" (LoRA merge at load dequantizes,
 * adds the delta and requantizes at group size 64, 4 bits; "File map":
 * lora.rs).  The pages state no rounding rule; this library's reading, per
 * group of 64 consecutive inputs of a row, in IEEE fp32:
 *   scale = bf16_rn((max - min) / (2^bits - 1)), bias = min (exact; a zero
 *   minimum is stored as +0), code = clamp(rint((w - bias) / scale), 0,
 *   2^bits - 1), round half to even, and code = 0 when scale == 0.
 * So dequantizing gives back w within scale/2 + (2^bits - 1)|scale - (max -
 * min)/(2^bits - 1)| per input.
 *   w       bf16 [N, K] row-major (device), 16-byte aligned, finite values.
 *   wq      out uint32 [N, K*bits/32]: codes lowest bits first (as read by
 *           the projections); 16-byte aligned.
 *   scales, biases  out bf16 [N, K/64]; 2-byte aligned.
 *   bits 4 or 8, group 64, K a positive multiple of 64 (<= 2^20), N >= 0.
 * The caller owns every buffer; the kernel runs on `stream`.  Errors:
 * GWA_ERR_UNSUPPORTED (bits, group), GWA_ERR_INVALID_ARG (shape, null),
 * GWA_ERR_MISALIGNED; nothing is enqueued on error. */
int gwa_quantize_affine(const uint16_t *w, int64_t N, int64_t K, int32_t bits,
                        int32_t group, uint32_t *wq, uint16_t *scales,
                        uint16_t *biases, void *stream);

/* Text of the last error raised on this thread ("" if none). */
const char *gwa_last_error(void);

/* Pipeline health.  The streaming and tensor-core kernels bound every wait
 * on their shared-memory pipelines (2 s); a wait that runs out is counted on
 * the device and the kernel returns early instead of hanging (its outputs
 * are then undefined).  Writes the count of such timeouts on the current
 * device since the last reset to *timeouts, and clears it if `reset`.
 * Synchronizes the current device (a diagnostics call, not for hot loops). */
int gwa_pipeline_status(uint32_t *timeouts, int32_t reset);

/* Test exports.  codes[N, K] (uint8) = q[n,k]; wf[N, K] (fp32) =
 * fmaf(scale, (float)q, bias): the dequantized weight rounded once to fp32.
 * Both are written on `stream`; the caller owns codes / wf. */
int gwa_debug_unpack(gwa_qweight w, uint8_t *codes, void *stream);
int gwa_debug_dequant(gwa_qweight w, float *wf, void *stream);

/* Test export: the kernels' bounded pipeline wait (see gwa_pipeline_status),
 * made to run out on purpose.  One CTA waits on a shared-memory barrier
 * that nothing completes, with `limit_us` microseconds (1 .. 2000000) in
 * place of the kernels' 2 s: warp 0 with the wait of the decode kernels,
 * warp 1 with the sleeping wait of the tensor-core kernel.  Writes the
 * device uint32 out[4] (16 bytes, caller-owned, 4-byte aligned): out[0],
 * out[2] = 1 when the respective wait gave up, out[1], out[3] = the
 * microseconds it waited.  The kernel returns normally, so the context
 * stays usable; the production timeout counters are not touched.
 * Errors: GWA_ERR_INVALID_ARG (limit, null), GWA_ERR_MISALIGNED. */
int gwa_debug_bounded_wait(uint32_t limit_us, uint32_t *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* GWA_H_ */
