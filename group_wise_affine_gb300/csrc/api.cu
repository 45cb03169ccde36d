// C ABI of libgwa.so (declared in include/gwa.h): argument validation,
// kernel selection and launch.  Nothing here allocates, synchronizes or
// aborts; every problem becomes a status code plus a thread-local message.
#include <math.h>
#include <mutex>
#include <map>
#include <stdarg.h>
#include <stdio.h>
#include <string>
#include <tuple>

#include "../../include/gwa.h"
#include "internal.h"
#include "qmm.h"

namespace gwa {

static thread_local std::string g_last_error;

int set_error(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}
#define fail set_error

static int cuda_fail(cudaError_t e, const char *what) {
    return fail(GWA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static bool aligned(const void *p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// ------------------------------------------------------------ device info
static std::mutex g_mu;

static int current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    return GWA_OK;
}

int num_sms() {
    static std::map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n;
    return n;
}

// The kernels are built for sm_103a only.
static int check_device() {
    static std::map<int, int> ok;
    int dev = 0;
    int rc = current_device(&dev);
    if (rc) return rc;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = ok.find(dev);
        if (it != ok.end())
            return it->second ? GWA_OK
                              : fail(GWA_ERR_CUDA, "device %d is not sm_103", dev);
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    const bool good = major == 10 && minor == 3;
    std::lock_guard<std::mutex> lk(g_mu);
    ok[dev] = good;
    return good ? GWA_OK
                : fail(GWA_ERR_CUDA, "device %d has compute capability %d.%d; "
                       "this library is built for sm_103a", dev, major, minor);
}

cudaError_t occupancy_grid(const void *kernel, int threads, size_t smem,
                           int *grid) {
    static std::map<std::tuple<int, const void *, size_t, int>, int> cache;
    static std::map<std::pair<int, const void *>, bool> attr_set;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = num_sms();
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(dev, kernel, smem, threads);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *grid = it->second;
        return cudaSuccess;
    }
    if (!attr_set[std::make_pair(dev, kernel)]) {
        // dynamic + static shared memory must stay within the opt-in limit
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin,
                                   cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        const int maxdyn = optin - (int)fa.sharedSizeBytes;
        if (maxdyn <= 0) return cudaErrorInvalidValue;
        e = cudaFuncSetAttribute(kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 maxdyn);
        if (e != cudaSuccess) return e;
        attr_set[std::make_pair(dev, kernel)] = true;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads,
                                                      smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    *grid = per_sm * sms;
    cache[key] = *grid;
    return cudaSuccess;
}

// Clusters of `cl` CTAs of `kernel` (`threads` threads, `smem` bytes of
// dynamic shared memory each) that the GPU keeps resident at once, 0 if it
// cannot launch them; cached per device, kernel, cluster size, block and
// shared memory.  The kernel's shared-memory attribute must be set first
// (occupancy_grid does).
int resident_clusters(const void *kernel, int cl, int threads, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int, int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, kernel, cl, threads, smem);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cl * (num_sms() / cl)));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = n;
    return n;
}

// Largest shared-memory carveout for a kernel whose CTAs (about 110 KB each)
// must sit two to an SM: the next kernel's CTA then starts beside this
// one's (programmatic dependent launch) instead of waiting for the SM to
// drain and reconfigure.
cudaError_t prefer_max_shared(const void *kernel) {
    static std::map<std::pair<int, const void *>, bool> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(dev, kernel);
    if (done[key]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) done[key] = true;
    return e;
}

// ------------------------------------------------------------ validation
// The tuned kernels take u4/u8 codes in groups of 64; the other widths and
// group sizes run on the general-format decode kernel.
static bool tuned_format(int bits, int group) {
    return (bits == 4 || bits == 8) && group == 64;
}

static_assert(GWA_FP8_E4M3 == kFp8, "fp8 format tag");

static int check_qweight(const gwa_qweight &w, const char *fn) {
    if (w.bits != 2 && w.bits != 3 && w.bits != 4 && w.bits != 6 &&
        w.bits != 8 && w.bits != GWA_FP8_E4M3)
        return fail(GWA_ERR_UNSUPPORTED,
                    "%s: bits=%d (supported: 2, 3, 4, 6, 8, GWA_FP8_E4M3)", fn,
                    (int)w.bits);
    if (w.group != 32 && w.group != 64 && w.group != 128)
        return fail(GWA_ERR_UNSUPPORTED,
                    "%s: group=%d (supported: 32, 64, 128)", fn, (int)w.group);
    if (w.N < 0 || w.K <= 0 || w.K % w.group != 0 || w.K % 64 != 0)
        return fail(GWA_ERR_INVALID_ARG,
                    "%s: N=%lld K=%lld (need N >= 0, K a positive multiple "
                    "of 64 and of the group)", fn, (long long)w.N,
                    (long long)w.K);
    if (w.K > (1 << 20))
        return fail(GWA_ERR_INVALID_ARG, "%s: K=%lld exceeds 2^20", fn,
                    (long long)w.K);
    if (w.N > 0 && (!w.wq || !w.scales || !w.biases))
        return fail(GWA_ERR_INVALID_ARG, "%s: null weight pointer", fn);
    if (!aligned(w.wq, 16))
        return fail(GWA_ERR_MISALIGNED, "%s: wq must be 16-byte aligned", fn);
    if (!aligned(w.scales, 2) || !aligned(w.biases, 2))
        return fail(GWA_ERR_MISALIGNED,
                    "%s: scales/biases must be 2-byte aligned", fn);
    return GWA_OK;
}

static int check_x(const uint16_t *x, int64_t M, const char *fn) {
    if (M < 0) return fail(GWA_ERR_INVALID_ARG, "%s: M=%lld", fn, (long long)M);
    if (M > 0 && !x) return fail(GWA_ERR_INVALID_ARG, "%s: null x", fn);
    if (!aligned(x, 16))
        return fail(GWA_ERR_MISALIGNED, "%s: x must be 16-byte aligned", fn);
    return GWA_OK;
}

static DenseParams dense_base(const uint16_t *x, int64_t M,
                              const gwa_qweight &w) {
    DenseParams p{};
    p.x = x;
    p.M = (int)M;
    p.K = (int)w.K;
    p.bits = w.bits;
    p.wq = w.wq;
    p.sc = w.scales;
    p.bi = w.biases;
    p.N = w.N;
    p.nch = (int)(w.K * code_bits(w.bits) / 128);
    p.group = (int)w.group;
    p.G = (int)(w.K / w.group);
    return p;
}

// Runs the decode kernels over token passes that fit in shared memory.
static int run_dense(int mode, DenseParams p, int64_t M, int64_t out_stride,
                     const int64_t *sec_sizes, cudaStream_t st,
                     const char *fn) {
    const bool generic = !tuned_format(p.bits, p.group);
    int mt = generic ? generic_max_tokens() : dense_max_tokens(p.bits, p.nch);
    if (mt < 1)
        return fail(GWA_ERR_INVALID_ARG, "%s: K=%d too large for staging", fn,
                    p.K);
    // The streaming kernel (up to four tokens a pass) outruns the staged one
    // even when it has to stream the weights twice for 5..8 tokens.
    if (!generic) {
        DenseParams probe = p;
        probe.M = 1;
        if (stream_eligible(probe)) mt = mt < 4 ? mt : 4;
    }
    // 5..8 tokens: the tensor-core decode kernel in one pass when the shape
    // allows it (the streaming kernel would stream the weights twice; at 2..4
    // tokens the two run level, and the streaming kernel stays)
    if (!generic && M >= 5 && M <= 8) {
        DenseParams q = p;
        q.M = (int)M;
        bool used = false;
        cudaError_t e = launch_mma(mode, q, st, &used);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        if (used) return GWA_OK;
    }
    for (int64_t t0 = 0; t0 < M; t0 += mt) {
        DenseParams q = p;
        q.M = (int)((M - t0) < mt ? (M - t0) : mt);
        q.x = p.x + t0 * p.K;
        if (mode == 3) {
            q.rope_pos = p.rope_pos + t0;
            q.rope_cs = p.rope_cs + t0 * (p.rope_hd / 2);
        }
        if (mode == 1 || mode == 3) {
            for (int s = 0; s < p.nsec; ++s)
                q.sec_out[s] = p.sec_out[s] ? p.sec_out[s] + t0 * sec_sizes[s]
                                            : nullptr;
        } else {
            q.y = p.y + t0 * out_stride;
        }
        bool used = false;
        if (generic) {
            // one token of u4 / u8 codes in groups of 32 or 128: the
            // chunk-per-lane kernel when the shape allows it; fp8 codes in
            // groups of 64: the streaming kernel (fp32 products)
            cudaError_t e = launch_group(mode, q, st, &used);
            if (e == cudaSuccess && !used && q.bits == kFp8)
                e = launch_stream(mode, q, st, &used);
            if (e == cudaSuccess && !used) e = launch_generic(mode, q, st);
            if (e != cudaSuccess) return cuda_fail(e, fn);
            continue;
        }
        cudaError_t e = launch_group(mode, q, st, &used);
        if (e == cudaSuccess && !used) e = launch_stream(mode, q, st, &used);
        if (e == cudaSuccess && !used) e = launch_dense(mode, q, st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    return GWA_OK;
}

// M > 8: the tensor-core kernel when the shape allows it, else the decode
// kernels in passes of up to eight tokens.  The workspace contract is the
// same either way.
static int run_prefill(const QmmArgs &a, int mode, const DenseParams &p,
                       int64_t out_stride, const int64_t *sec_sizes,
                       void *workspace, size_t workspace_bytes,
                       cudaStream_t st, const char *fn) {
    if (qmm_eligible(a)) return qmm_run(a, workspace, workspace_bytes, st);
    const size_t need = qmm_workspace_bytes(a.M, a.w.K);
    if (!workspace || workspace_bytes < need)
        return fail(GWA_ERR_WORKSPACE,
                    "%s: M=%lld K=%lld needs %zu bytes of workspace (got %zu)",
                    fn, (long long)a.M, (long long)a.w.K, need,
                    workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return fail(GWA_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned",
                    fn);
    // the decode kernels raise no status: the word reads 0 after the call,
    // as after a tensor-core call that met no problem
    const cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return run_dense(mode, p, a.M, out_stride, sec_sizes, st, fn);
}

}  // namespace gwa

using namespace gwa;

extern "C" {

const char *gwa_last_error(void) { return g_last_error.c_str(); }

int gwa_pipeline_status(uint32_t *timeouts, int32_t reset) {
    g_last_error.clear();
    if (!timeouts) return fail(GWA_ERR_INVALID_ARG, "gwa_pipeline_status: null");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "gwa_pipeline_status");
    *timeouts = group_timeouts(reset != 0) + stream_timeouts(reset != 0) +
                moe_stream_timeouts(reset != 0) + qmm_timeouts(reset != 0) +
                mma_timeouts(reset != 0);
    e = cudaGetLastError();
    return e == cudaSuccess ? GWA_OK : cuda_fail(e, "gwa_pipeline_status");
}

size_t gwa_workspace_bytes(int64_t M, int64_t K) {
    if (M <= 8 || K <= 0) return 0;
    return qmm_workspace_bytes(M, K);
}

int gwa_qmv_affine(const uint16_t *x, int64_t M, gwa_qweight w, uint16_t *y,
                   void *workspace, size_t workspace_bytes, void *stream) {
    const char *fn = "gwa_qmv_affine";
    g_last_error.clear();
    int rc = check_qweight(w, fn);
    if (!rc) rc = check_x(x, M, fn);
    if (rc) return rc;
    if (M == 0 || w.N == 0) return GWA_OK;
    if (!y) return fail(GWA_ERR_INVALID_ARG, "%s: null y", fn);
    if (!aligned(y, 2)) return fail(GWA_ERR_MISALIGNED, "%s: y alignment", fn);
    if ((rc = check_device())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DenseParams p = dense_base(x, M, w);
    p.y = y;
    if (M > 8) {
        QmmArgs a{};
        a.x = x; a.M = M; a.w = w; a.mode = 0; a.y = y;
        return run_prefill(a, 0, p, w.N, nullptr, workspace, workspace_bytes,
                           st, fn);
    }
    return run_dense(0, p, M, w.N, nullptr, st, fn);
}

int gwa_qmv_fused_sections(const uint16_t *x, int64_t M, gwa_qweight w,
                           int32_t n_sections, const int64_t *section_sizes,
                           uint16_t *const *outs,
                           const uint16_t *const *out_bias, void *workspace,
                           size_t workspace_bytes, void *stream) {
    const char *fn = "gwa_qmv_fused_sections";
    g_last_error.clear();
    int rc = check_qweight(w, fn);
    if (!rc) rc = check_x(x, M, fn);
    if (rc) return rc;
    if (n_sections < 1 || n_sections > kMaxSections)
        return fail(GWA_ERR_INVALID_ARG, "%s: n_sections=%d (1..%d)", fn,
                    (int)n_sections, kMaxSections);
    if (!section_sizes || !outs)
        return fail(GWA_ERR_INVALID_ARG, "%s: null section arrays", fn);
    int64_t total = 0;
    for (int s = 0; s < n_sections; ++s) {
        if (section_sizes[s] < 0)
            return fail(GWA_ERR_INVALID_ARG, "%s: section %d size %lld", fn, s,
                        (long long)section_sizes[s]);
        if (section_sizes[s] > 0 && M > 0 && !outs[s])
            return fail(GWA_ERR_INVALID_ARG, "%s: null output %d", fn, s);
        if (!aligned(outs[s], 2))
            return fail(GWA_ERR_MISALIGNED, "%s: output %d alignment", fn, s);
        if (out_bias && !aligned(out_bias[s], 2))
            return fail(GWA_ERR_MISALIGNED, "%s: bias %d alignment", fn, s);
        total += section_sizes[s];
    }
    if (total != w.N)
        return fail(GWA_ERR_INVALID_ARG,
                    "%s: section sizes add up to %lld, weight has %lld rows",
                    fn, (long long)total, (long long)w.N);
    if (M == 0 || w.N == 0) return GWA_OK;
    if ((rc = check_device())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DenseParams p = dense_base(x, M, w);
    p.nsec = n_sections;
    p.sec_start[0] = 0;
    for (int s = 0; s < n_sections; ++s) {
        p.sec_start[s + 1] = p.sec_start[s] + section_sizes[s];
        p.sec_out[s] = outs[s];
        p.sec_bias[s] = out_bias ? out_bias[s] : nullptr;
    }
    if (M > 8) {
        QmmArgs a{};
        a.x = x; a.M = M; a.w = w; a.mode = 1;
        a.nsec = n_sections;
        for (int s = 0; s <= n_sections; ++s) a.sec_start[s] = p.sec_start[s];
        for (int s = 0; s < n_sections; ++s) {
            a.sec_out[s] = p.sec_out[s];
            a.sec_bias[s] = p.sec_bias[s];
        }
        return run_prefill(a, 1, p, 0, section_sizes, workspace,
                           workspace_bytes, st, fn);
    }
    return run_dense(1, p, M, 0, section_sizes, st, fn);
}

int gwa_qmv_qkv_rope(const uint16_t *x, int64_t M, gwa_qweight w,
                     int64_t q_size, int64_t kv_size, int32_t head_dim,
                     double rope_base, const int32_t *positions, uint16_t *q,
                     uint16_t *k, uint16_t *v,
                     const uint16_t *const *out_bias, void *workspace,
                     size_t workspace_bytes, void *stream) {
    const char *fn = "gwa_qmv_qkv_rope";
    g_last_error.clear();
    int rc = check_qweight(w, fn);
    if (!rc) rc = check_x(x, M, fn);
    if (rc) return rc;
    if (head_dim < 2 || head_dim % 2 != 0 || head_dim > 256)
        return fail(GWA_ERR_INVALID_ARG, "%s: head_dim=%d (even, 2..256)", fn,
                    (int)head_dim);
    if (q_size < 0 || kv_size < 0 || q_size % head_dim != 0 ||
        kv_size % head_dim != 0)
        return fail(GWA_ERR_INVALID_ARG,
                    "%s: q_size=%lld kv_size=%lld (multiples of head_dim)", fn,
                    (long long)q_size, (long long)kv_size);
    if (q_size + 2 * kv_size != w.N)
        return fail(GWA_ERR_INVALID_ARG,
                    "%s: q_size + 2*kv_size = %lld, weight has %lld rows", fn,
                    (long long)(q_size + 2 * kv_size), (long long)w.N);
    if (w.N >= ((int64_t)1 << 30))
        return fail(GWA_ERR_INVALID_ARG, "%s: N=%lld (< 2^30)", fn,
                    (long long)w.N);
    if (!(rope_base > 0.0) || rope_base > 1e30)
        return fail(GWA_ERR_INVALID_ARG, "%s: rope_base=%g", fn, rope_base);
    uint16_t *outs[3] = {q, k, v};
    const int64_t sizes[3] = {q_size, kv_size, kv_size};
    for (int s = 0; s < 3; ++s) {
        if (sizes[s] > 0 && M > 0 && !outs[s])
            return fail(GWA_ERR_INVALID_ARG, "%s: null output %d", fn, s);
        if (!aligned(outs[s], 2))
            return fail(GWA_ERR_MISALIGNED, "%s: output %d alignment", fn, s);
        if (out_bias && !aligned(out_bias[s], 2))
            return fail(GWA_ERR_MISALIGNED, "%s: bias %d alignment", fn, s);
    }
    if (M > 0 && !positions)
        return fail(GWA_ERR_INVALID_ARG, "%s: null positions", fn);
    if (!aligned(positions, 4))
        return fail(GWA_ERR_MISALIGNED, "%s: positions alignment", fn);
    if (M == 0 || w.N == 0) return GWA_OK;
    if ((rc = check_device())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DenseParams p = dense_base(x, M, w);
    p.nsec = 3;
    p.sec_start[0] = 0;
    for (int s = 0; s < 3; ++s) {
        p.sec_start[s + 1] = p.sec_start[s] + sizes[s];
        p.sec_out[s] = outs[s];
        p.sec_bias[s] = out_bias ? out_bias[s] : nullptr;
    }
    DenseParams r = p;
    r.rope_hd = head_dim;
    r.rope_end = q_size + kv_size;
    r.rope_pos = positions;
    r.rope_r = pow(rope_base, -2.0 / (double)head_dim);
    if (M == 1 && (w.bits == 4 || w.bits == 8) &&
        (w.group == 32 || w.group == 64 || w.group == 128)) {
        // the one-token kernel forms its own (cos, sin) and rotates Q and K
        // in its epilogue
        bool used = false;
        cudaError_t e = launch_group(3, r, st, &used);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        if (used) return GWA_OK;
    }
    // otherwise a (cos, sin) table in the workspace (after the tensor-core
    // path's area), then the kernels rotate in their epilogues
    const size_t need = gwa_qkv_rope_workspace_bytes(M, w.K, head_dim);
    if (!workspace || workspace_bytes < need)
        return fail(GWA_ERR_WORKSPACE,
                    "%s: M=%lld K=%lld head_dim=%d needs %zu bytes of workspace "
                    "(got %zu)", fn, (long long)M, (long long)w.K, (int)head_dim,
                    need, workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return fail(GWA_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned",
                    fn);
    const size_t qmm_area = M > 8 ? (qmm_workspace_bytes(M, w.K) + 255) / 256 * 256 : 0;
    float2 *cs = reinterpret_cast<float2 *>(static_cast<unsigned char *>(workspace) +
                                            qmm_area);
    cudaError_t e = launch_rope_table(cs, M, head_dim, r.rope_r, positions, st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    r.rope_cs = cs;
    if (M > 8) {
        // the status word reads 0 after a call that met no problem, on the
        // decode kernels as on the tensor cores
        e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        // tensor cores when the shape allows it and each head and section
        // is whole inside the 128-row tiles
        QmmArgs a{};
        a.x = x; a.M = M; a.w = w; a.mode = 3;
        a.nsec = 3;
        for (int s = 0; s <= 3; ++s) a.sec_start[s] = p.sec_start[s];
        for (int s = 0; s < 3; ++s) {
            a.sec_out[s] = p.sec_out[s];
            a.sec_bias[s] = p.sec_bias[s];
        }
        a.rope_hd = head_dim;
        a.rope_end = q_size + kv_size;
        a.rope_cs = cs;
        if (qmm_eligible(a) && 128 % head_dim == 0 && q_size % 128 == 0 &&
            kv_size % 128 == 0)
            return qmm_run(a, workspace, workspace_bytes, st);
    }
    return run_dense(3, r, M, 0, sizes, st, fn);
}

size_t gwa_qkv_rope_workspace_bytes(int64_t M, int64_t K, int32_t head_dim) {
    if (M < 1 || head_dim < 2 || K < 1) return 0;
    const size_t qmm_area = M > 8 ? (qmm_workspace_bytes(M, K) + 255) / 256 * 256 : 0;
    const size_t b = (size_t)M * (size_t)(head_dim / 2) * 8;
    return qmm_area + (b + 255) / 256 * 256;
}

int gwa_qmv_gate_up_silu(const uint16_t *x, int64_t M, gwa_qweight w,
                         uint16_t *h, void *workspace, size_t workspace_bytes,
                         void *stream) {
    const char *fn = "gwa_qmv_gate_up_silu";
    g_last_error.clear();
    int rc = check_qweight(w, fn);
    if (!rc) rc = check_x(x, M, fn);
    if (rc) return rc;
    if (w.N % 2 != 0)
        return fail(GWA_ERR_INVALID_ARG, "%s: N=%lld must be even (gate; up)",
                    fn, (long long)w.N);
    if (M == 0 || w.N == 0) return GWA_OK;
    if (!h) return fail(GWA_ERR_INVALID_ARG, "%s: null h", fn);
    if (!aligned(h, 2)) return fail(GWA_ERR_MISALIGNED, "%s: h alignment", fn);
    if ((rc = check_device())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DenseParams p = dense_base(x, M, w);
    p.y = h;
    p.I = w.N / 2;
    if (M > 8) {
        QmmArgs a{};
        a.x = x; a.M = M; a.w = w; a.mode = 2; a.y = h;
        return run_prefill(a, 2, p, w.N / 2, nullptr, workspace,
                           workspace_bytes, st, fn);
    }
    return run_dense(2, p, M, w.N / 2, nullptr, st, fn);
}

int gwa_moe_qmv_gather(const uint16_t *x, int64_t M, int32_t topk,
                       const int32_t *expert_ids, const float *route_w,
                       gwa_qweight w, int32_t num_experts, int32_t mode,
                       uint16_t *out, int32_t *status, void *stream) {
    const char *fn = "gwa_moe_qmv_gather";
    g_last_error.clear();
    int rc = check_qweight(w, fn);
    if (!rc) rc = check_x(x, M, fn);
    if (rc) return rc;
    if (mode != GWA_MOE_GATE_UP_SILU && mode != GWA_MOE_DOWN_COMBINE)
        return fail(GWA_ERR_INVALID_ARG, "%s: mode=%d", fn, (int)mode);
    if (!tuned_format(w.bits, w.group))
        return fail(GWA_ERR_UNSUPPORTED,
                    "%s: bits=%d group=%d (experts: u4 or u8, group 64)", fn,
                    (int)w.bits, (int)w.group);
    if (M > 8)
        return fail(GWA_ERR_UNSUPPORTED, "%s: M=%lld (decode path: M <= 8)", fn,
                    (long long)M);
    if (topk < 1 || topk > 32)
        return fail(GWA_ERR_INVALID_ARG, "%s: topk=%d (1..32)", fn, (int)topk);
    if (num_experts < 1)
        return fail(GWA_ERR_INVALID_ARG, "%s: num_experts=%d", fn,
                    (int)num_experts);
    if (mode == GWA_MOE_GATE_UP_SILU && w.N % 2 != 0)
        return fail(GWA_ERR_INVALID_ARG, "%s: gate+up rows per expert must be "
                    "even", fn);
    if (M == 0 || w.N == 0) return GWA_OK;
    if (!expert_ids || !out)
        return fail(GWA_ERR_INVALID_ARG, "%s: null ids or output", fn);
    if (mode == GWA_MOE_DOWN_COMBINE && !route_w)
        return fail(GWA_ERR_INVALID_ARG, "%s: down mode needs route_w", fn);
    if (!aligned(expert_ids, 4) || !aligned(route_w, 4) ||
        !aligned(status, 4) || !aligned(out, 2))
        return fail(GWA_ERR_MISALIGNED, "%s: ids/route_w/status/out alignment",
                    fn);
    const int nch = (int)(w.K * w.bits / 128);
    if ((rc = check_device())) return rc;
    MoeParams p{};
    p.x = x;
    p.M = (int)M;
    p.topk = topk;
    p.K = (int)w.K;
    p.bits = w.bits;
    p.ids = expert_ids;
    p.route_w = route_w;
    p.wq = w.wq;
    p.sc = w.scales;
    p.bi = w.biases;
    p.N = w.N;
    p.E = num_experts;
    p.nch = nch;
    p.G = (int)(w.K / 64);
    p.out = out;
    p.status = status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool used = false;
    cudaError_t e = launch_moe_stream(mode, p, st, &used);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (used) return GWA_OK;
    // rows longer than the streaming kernel handles: staged kernels
    const int cap = moe_max_tokens(w.bits, nch, mode);
    if ((mode == 0 && cap < 1) || (mode == 1 && cap < M * topk))
        return fail(GWA_ERR_UNSUPPORTED,
                    "%s: M*topk=%lld inputs of K=%lld do not fit in shared "
                    "memory", fn, (long long)(M * topk), (long long)w.K);
    e = mode == GWA_MOE_GATE_UP_SILU ? launch_moe_gate_up(p, st)
                                     : launch_moe_down(p, st);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return GWA_OK;
}

int gwa_debug_unpack(gwa_qweight w, uint8_t *codes, void *stream) {
    const char *fn = "gwa_debug_unpack";
    g_last_error.clear();
    int rc = check_qweight(w, fn);
    if (rc) return rc;
    if (w.N == 0) return GWA_OK;
    if (!codes) return fail(GWA_ERR_INVALID_ARG, "%s: null codes", fn);
    if ((rc = check_device())) return rc;
    cudaError_t e = launch_debug_unpack(w.wq, w.N, w.K, w.bits, codes,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GWA_OK : cuda_fail(e, fn);
}

int gwa_quantize_affine(const uint16_t *w, int64_t N, int64_t K, int32_t bits,
                        int32_t group, uint32_t *wq, uint16_t *scales,
                        uint16_t *biases, void *stream) {
    const char *fn = "gwa_quantize_affine";
    g_last_error.clear();
    // the output weight's checks are the projections' (bits, group, shape,
    // alignment of wq / scales / biases)
    const gwa_qweight out{wq, scales, biases, N, K, bits, group};
    int rc = check_qweight(out, fn);
    if (rc) return rc;
    if (!tuned_format(bits, group))
        return fail(GWA_ERR_UNSUPPORTED,
                    "%s: bits=%d group=%d (quantization: u4 or u8, group 64)",
                    fn, (int)bits, (int)group);
    if (N == 0) return GWA_OK;
    if (!w) return fail(GWA_ERR_INVALID_ARG, "%s: null w", fn);
    if (!aligned(w, 16))
        return fail(GWA_ERR_MISALIGNED, "%s: w must be 16-byte aligned", fn);
    if ((rc = check_device())) return rc;
    cudaError_t e = launch_quantize(w, N, K, bits, wq, scales, biases,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GWA_OK : cuda_fail(e, fn);
}

static int check_attention(int64_t B, int32_t Hq, int32_t Lq, int32_t D,
                           int32_t Hkv, int64_t T, int32_t bits, int32_t group,
                           int32_t causal, const char *fn) {
    if (D != 64 && D != 128 && D != 256)
        return fail(GWA_ERR_UNSUPPORTED, "%s: D=%d (64, 128 or 256)", fn, (int)D);
    if ((bits != 4 && bits != 8) || group != 64)
        return fail(GWA_ERR_UNSUPPORTED,
                    "%s: bits=%d group=%d (values: u4 or u8, group 64)", fn,
                    (int)bits, (int)group);
    if (B < 0 || B > 65535 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || Lq < 0 ||
        T < 1 || T > 0x7fffffffLL || (int64_t)Hkv * ((Hq / Hkv * (int64_t)Lq + 7) / 8) > 65535)
        return fail(GWA_ERR_INVALID_ARG,
                    "%s: B=%lld Hq=%d Hkv=%d Lq=%d T=%lld", fn, (long long)B,
                    (int)Hq, (int)Hkv, (int)Lq, (long long)T);
    if (causal && Lq > T)
        return fail(GWA_ERR_INVALID_ARG,
                    "%s: causal with Lq=%d > T=%lld (every query must see a key)",
                    fn, (int)Lq, (long long)T);
    return GWA_OK;
}

int gwa_sdpa_dequant_v(const uint16_t *q, int64_t B, int32_t Hq, int32_t Lq,
                       int32_t D, const uint16_t *k, int32_t Hkv, int64_t T,
                       const uint32_t *vq, const uint16_t *vs,
                       const uint16_t *vb, int32_t bits, int32_t group,
                       float scale, int32_t causal, uint16_t *out,
                       void *workspace, size_t workspace_bytes, void *stream) {
    const char *fn = "gwa_sdpa_dequant_v";
    g_last_error.clear();
    int rc = check_attention(B, Hq, Lq, D, Hkv, T, bits, group, causal, fn);
    if (rc) return rc;
    if (B == 0 || Lq == 0) return GWA_OK;
    if (!q || !k || !vq || !vs || !vb || !out)
        return fail(GWA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(vq, 8) || !aligned(vs, 8) ||
        !aligned(vb, 8) || !aligned(out, 2))
        return fail(GWA_ERR_MISALIGNED,
                    "%s: alignment (q, k 16 bytes; codes, scales, biases 8)", fn);
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
        return fail(GWA_ERR_INVALID_ARG, "%s: scale", fn);
    const size_t need = gwa_sdpa_workspace_bytes(B, Hq, Hkv, Lq, T, D);
    if (!workspace || workspace_bytes < need)
        return fail(GWA_ERR_WORKSPACE, "%s: needs %zu bytes of workspace (got %zu)",
                    fn, need, workspace_bytes);
    if (!aligned(workspace, 16))
        return fail(GWA_ERR_MISALIGNED, "%s: workspace alignment", fn);
    if ((rc = check_device())) return rc;
    cudaError_t e = launch_attention(q, k, vq, vs, vb, out,
                                     static_cast<float *>(workspace), (int)B,
                                     Hq, Hkv, Lq, (int)T, D, bits, scale,
                                     causal ? 1 : 0,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GWA_OK : cuda_fail(e, fn);
}

size_t gwa_sdpa_workspace_bytes(int64_t B, int32_t Hq, int32_t Hkv, int32_t Lq,
                                int64_t T, int32_t D) {
    if (B < 1 || Hkv < 1 || Hq < Hkv || Lq < 1 || T < 1 || D < 1 ||
        T > 0x7fffffffLL)
        return 0;
    return attention_workspace_bytes((int)B, Hq, Hkv, Lq, (int)T, D);
}

int gwa_debug_bounded_wait(uint32_t limit_us, uint32_t *out, void *stream) {
    const char *fn = "gwa_debug_bounded_wait";
    g_last_error.clear();
    if (limit_us < 1 || limit_us > 2000000u)
        return fail(GWA_ERR_INVALID_ARG, "%s: limit_us=%u (1 .. 2000000)", fn,
                    (unsigned)limit_us);
    if (!out) return fail(GWA_ERR_INVALID_ARG, "%s: null out", fn);
    if (!aligned(out, 4)) return fail(GWA_ERR_MISALIGNED, "%s: alignment", fn);
    int rc = check_device();
    if (rc) return rc;
    cudaError_t e = launch_debug_wait(out, 1000ull * limit_us,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GWA_OK : cuda_fail(e, fn);
}

int gwa_debug_dequant(gwa_qweight w, float *wf, void *stream) {
    const char *fn = "gwa_debug_dequant";
    g_last_error.clear();
    int rc = check_qweight(w, fn);
    if (rc) return rc;
    if (w.N == 0) return GWA_OK;
    if (!wf) return fail(GWA_ERR_INVALID_ARG, "%s: null output", fn);
    if (!aligned(wf, 4)) return fail(GWA_ERR_MISALIGNED, "%s: alignment", fn);
    if ((rc = check_device())) return rc;
    cudaError_t e = launch_debug_dequant(w.wq, w.scales, w.biases, w.N, w.K,
                                         w.bits, (int)w.group, wf,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GWA_OK : cuda_fail(e, fn);
}

}  // extern "C"
