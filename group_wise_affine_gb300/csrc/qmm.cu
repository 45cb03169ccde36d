// Prefill-shaped (M > 8) path.
#include "qmm.h"

namespace gwa {

size_t qmm_workspace_bytes(int64_t M, int64_t K) {
    (void)M;
    (void)K;
    return 0;
}

int qmm_run(const QmmArgs &a, void *workspace, size_t workspace_bytes,
            cudaStream_t st) {
    (void)a;
    (void)workspace;
    (void)workspace_bytes;
    (void)st;
    return set_error(GWA_ERR_UNSUPPORTED, "M > 8: tensor-core path not built");
}

}  // namespace gwa
