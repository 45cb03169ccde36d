// gwa_qmv_affine_noalloc: the plain projection for callers that cannot
// allocate device memory.  Some callers have no device allocator at hand or
// must not allocate on this path -- for example a plug-in inside a host
// framework that owns all device memory, or a serving loop that cannot afford
// an allocation call (it may synchronize the device, or fail under memory
// pressure in the middle of a request).  Such callers cannot provide the
// workspace that the tensor-core path (M > 8) needs, so this entry point uses
// a fixed scratch buffer that lives in the library itself.
//
// The scratch is a file-scope device array.  In host code its name is only a
// host-side stand-in, not a device address, so every call looks up the
// device address on the current device with cudaGetSymbolAddress (no
// allocation, no synchronization) and hands it to the kernels as their
// workspace.  Looking it up per call rather than caching it keeps the address
// right after the device's context is torn down and made again.
#include "../../include/gwa.h"
#include "qmm.h"

namespace gwa {

// Modest on purpose: every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[GWA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch on the current device.
static int noalloc_scratch(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
        return set_error(GWA_ERR_CUDA,
                         "gwa_qmv_affine_noalloc: scratch lookup failed: %s",
                         cudaGetErrorString(e));
    *out = p;
    return GWA_OK;
}

}  // namespace gwa

extern "C" int gwa_qmv_affine_noalloc(const uint16_t *x, int64_t M,
                                      gwa_qweight w, uint16_t *y,
                                      void *stream) {
    // M <= 8 runs the decode kernels, which need no scratch at all.
    if (M <= 8) return gwa_qmv_affine(x, M, w, y, nullptr, 0, stream);
    const size_t need = gwa_workspace_bytes(M, w.K);
    if (need > (size_t)GWA_NOALLOC_SCRATCH_BYTES)
        return gwa::set_error(
            GWA_ERR_WORKSPACE,
            "gwa_qmv_affine_noalloc: M=%lld K=%lld needs %zu bytes of scratch; "
            "the built-in scratch holds %zu (use gwa_qmv_affine with a "
            "workspace)",
            (long long)M, (long long)w.K, need,
            (size_t)GWA_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    int rc = gwa::noalloc_scratch(&scratch);
    if (rc) return rc;
    return gwa_qmv_affine(x, M, w, y, scratch, GWA_NOALLOC_SCRATCH_BYTES,
                          stream);
}
