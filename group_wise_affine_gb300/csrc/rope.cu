// Table of rotary-embedding (cos, sin) pairs for one call of the fused QKV
// projection with RoPE: cs[m * d/2 + i] for token m and pair index i of a
// head of d, t = positions[m] * base^(-2i/d) ("The Cathedral Doubled
// Itself", "The kernel that worked and the kernel that won't": RoPE on the
// materialized Q and K; the form is the textbook rotate-half one).  The
// projection kernels for more than one token read it in their epilogues and
// rotate the fp32 results before rounding to bf16 (rotating the rounded
// outputs would leave errors relative to the inputs' magnitude, above the
// output tolerance where the rotated value is small).  Each entry's angle is
// formed in fp64 from r = base^(-2/d) (see rope_cos_sin); the table is
// formed once per token and frequency, not per head, because fp64 is slow
// on this GPU.
#include "common.cuh"
#include "internal.h"

namespace gwa {

__global__ void __launch_bounds__(256)
    rope_table_kernel(float2 *__restrict__ cs, int64_t entries, int d,
                      double r, const int32_t *__restrict__ positions) {
    if (threadIdx.x == 0) pdl_launch_dependents();
    // positions are an input no kernel of this library writes, so the first
    // entry's (slow, fp64) angle is formed before the wait; the stores wait,
    // since the previous kernel may still read this workspace
    const int half = d / 2;
    int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    float2 v = make_float2(1.0f, 0.0f);
    if (e < entries)
        v = rope_cos_sin(positions[e / half], (int)(e % half), r);
    pdl_wait_primary();
    if (e < entries) cs[e] = v;
    for (e += step; e < entries; e += step)
        cs[e] = rope_cos_sin(positions[e / half], (int)(e % half), r);
}

cudaError_t launch_rope_table(float2 *cs, int64_t M, int head_dim, double r,
                              const int32_t *positions, cudaStream_t st) {
    const int64_t entries = M * (head_dim / 2);
    if (entries <= 0) return cudaSuccess;
    int64_t grid = (entries + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (grid > cap) grid = cap;
    return launch_pdl(reinterpret_cast<const void *>(rope_table_kernel),
                      (unsigned)grid, 256u, 0, st, cs, entries, head_dim, r,
                      positions);
}

}  // namespace gwa
