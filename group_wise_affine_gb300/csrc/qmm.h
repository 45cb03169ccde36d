// Prefill-shaped (M > 8) path: tensor-core (tcgen05) kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gwa.h"
#include "internal.h"

namespace gwa {

struct QmmArgs {
    const uint16_t *x;  // [M, K] bf16
    int64_t M;
    gwa_qweight w;
    int mode;           // 0 plain, 1 sections, 2 gate+up SwiGLU,
                        // 3 sections with the rotary embedding
    uint16_t *y;        // plain: [M, N]; gate+up: [M, N/2]
    int nsec;
    int64_t sec_start[kMaxSections + 1];
    uint16_t *sec_out[kMaxSections];
    const uint16_t *sec_bias[kMaxSections];
    // mode 3: rows [0, rope_end) rotate in heads of rope_hd (dividing 128,
    // sections whole 128-row tiles) with (cos, sin) rope_cs[m * hd/2 + i]
    int rope_hd;
    int64_t rope_end;
    const float2 *rope_cs;
};

size_t qmm_workspace_bytes(int64_t M, int64_t K);
// Whether the tensor-core kernel takes this shape (K a multiple of 512,
// 16-byte aligned weights); otherwise M > 8 runs on the decode kernels in
// passes of up to eight tokens.
bool qmm_eligible(const QmmArgs &a);
int qmm_run(const QmmArgs &a, void *workspace, size_t workspace_bytes,
            cudaStream_t st);

// Tensor-core pipeline waits that ran out of time (read, optionally reset).
unsigned int qmm_timeouts(bool reset);

// Records the thread's last error text and returns `code`.
int set_error(int code, const char *fmt, ...);

}  // namespace gwa
