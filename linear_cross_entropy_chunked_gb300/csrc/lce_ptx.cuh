// Inline-PTX helpers shared by the kernels of this library (sm_103a):
// mbarriers with bounded waits, the async-proxy fence, and the cluster
// primitives (rank, distributed shared-memory addresses, remote arrivals,
// cluster barrier).
//
// Every wait here is bounded by a wall-clock limit read from %globaltimer; on
// expiry the waiting CTA records FLAG_TIMEOUT in the workspace header and its
// later waits return false at once, so a kernel can leave cleanly instead of
// hanging the device.
#pragma once
#include "lce_internal.h"

namespace lce {

// ---------------------------------------------------------------- mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared abort word of the CTA: set by whichever thread's wait ran out first.
struct Abort {
    volatile int *flag_smem;
    int *hdr;
    uint64_t limit_ns;
};

// Bounded wait for the phase with the given parity. Returns false (and makes
// every later wait of the CTA return false at once) when the limit runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const Abort &ab) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (*ab.flag_smem) return false;
        if (global_timer_ns() - t0 > ab.limit_ns) {
            *ab.flag_smem = 1;
            atomicOr(ab.hdr + HDR_FLAG, FLAG_TIMEOUT);
            return false;
        }
    }
}

// Drain wait used on the abort path only: fixed bound, no flag update.
__device__ __forceinline__ void mbar_wait_drain(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

// Orders this CTA's generic-proxy shared-memory accesses before later
// async-proxy (TMA / bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cluster helpers

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait with cluster-scope acquire (for data another CTA wrote).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, const Abort &ab) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_cluster(a, parity)) return true;
        if (*ab.flag_smem) return false;
        if (global_timer_ns() - t0 > ab.limit_ns) {
            *ab.flag_smem = 1;
            atomicOr(ab.hdr + HDR_FLAG, FLAG_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

}  // namespace lce
