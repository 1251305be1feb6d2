// Thread-block cluster helpers (inline PTX, sm_103a): rank and size within the
// cluster, the cluster-wide barrier, and 32-bit loads from a peer CTA's shared
// memory (distributed shared memory). Used by the split-row forward kernel and
// the backward's dw reduction.
#pragma once

#include <stdint.h>

namespace rmsn {

static __device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

static __device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Cluster-wide barrier: release this CTA's prior shared-memory writes, acquire the
// peers'. Every thread of every CTA of the cluster must reach it; the .aligned
// forms need the whole warp converged, hence the __syncwarp.
static __device__ __forceinline__ void cluster_sync() {
    __syncwarp();
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}

// Reads a 32-bit word at the same shared-memory offset in CTA `rank` of the cluster.
static __device__ __forceinline__ uint32_t ld_peer_u32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

}  // namespace rmsn
