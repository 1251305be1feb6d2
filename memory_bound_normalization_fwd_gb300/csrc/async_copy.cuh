// Shared-memory barrier (mbarrier) and bulk asynchronous copy (TMA, non-tensor
// cp.async.bulk) helpers for the staged kernels, as inline PTX for sm_103a.
// Every wait is bounded: it polls against a clock64 deadline and reports
// failure instead of spinning forever.
#pragma once

#include <stdint.h>

namespace rmsn {

static __device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

static __device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

static __device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

static __device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy; completion is signalled on `bar` as `bytes` transactions.
static __device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Orders this thread's earlier generic-proxy writes to shared memory before later
// async-proxy (bulk copy) reads of them; each writing thread runs it before the
// barrier that precedes the copy.
static __device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared -> global bulk copy, tracked in the issuing thread's bulk async-groups.
// Both addresses 16-byte aligned, `bytes` a multiple of 16.
static __device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
}

static __device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Returns once every bulk group this thread committed has finished reading its
// shared-memory source (the buffer may then be overwritten).
static __device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Returns once at most the newest of this thread's committed bulk groups may
// still be reading its shared-memory source.
static __device__ __forceinline__ void bulk_wait_read_all_but_newest() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Returns once every bulk group this thread committed has completed (its global
// writes are done).
static __device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Asks for `bytes` of global memory at `src` to be brought into L2 (a hint:
// nothing lands in shared memory or registers and there is no completion to
// wait for). `src` 16-byte aligned, `bytes` a multiple of 16. A later load of
// those lines then meets L2 latency instead of DRAM latency.
static __device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

static __device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

static __device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most `limit` SM cycles.
static __device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (clock64() - t0 < limit) {
        if (mbar_try(bar, parity)) return true;
    }
    return false;
}

}  // namespace rmsn
