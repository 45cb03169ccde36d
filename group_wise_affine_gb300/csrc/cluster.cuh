// Thread-block cluster helpers shared by the kernels that combine partial
// sums across the CTAs of a cluster through distributed shared memory.
#pragma once

#include "common.cuh"

namespace gwa {

// Thread-block clusters: this CTA's rank, a barrier of every thread of the
// cluster (release / acquire), and a load from a peer's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release;\n"
        "barrier.cluster.wait.acquire;" ::
            : "memory");
}
// fp32 at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(const float *local,
                                                uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(a)
                 : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

// N fp32 values at local + j * stride (j < N), same offsets, in CTA `rank`
// of the cluster: one address mapping, then all N loads issued before any
// is used (each remote load's latency is long).
template <int N>
__device__ __forceinline__ void ld_cluster_f32_n(const float *local, uint32_t rank,
                                                 uint32_t stride, float (&v)[N]) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(a)
                 : "r"(smem_u32(local)), "r"(rank));
#pragma unroll
    for (int j = 0; j < N; ++j)
        asm volatile("ld.shared::cluster.f32 %0, [%1];"
                     : "=f"(v[j])
                     : "r"(a + (uint32_t)j * stride * 4u)
                     : "memory");
}

}  // namespace gwa
