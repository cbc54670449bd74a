// cluster.cuh -- inline-PTX wrappers for thread-block clusters and for handing data between
// the CTAs of a cluster through global memory (sm_103a): the CTA's rank, addresses in another
// CTA's shared memory, mbarrier arrivals on another CTA's barriers, waits that acquire at cluster
// scope, the generic-to-async proxy fence for global memory, a global-to-shared bulk copy and the
// cluster-wide barrier. Each wrapper is one documented PTX instruction (or a short fixed
// sequence), plus the bounded waits built on them.
#pragma once
#include <cstdint>

#include "kda_common.cuh"

namespace kda {

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The address of the same shared-memory location in cluster CTA `rank` (a shared::cluster address).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of any CTA of the cluster, with no memory ordering of its own: a release
// is formed by fence_acq_rel_cluster() before it. (A release-qualified arrive fences on every
// arrival, which costs about half a microsecond each.)
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Acquire-release fence at cluster scope: with the relaxed arrivals after it, a release of
// everything this thread has written or observed (through a CTA barrier, the writes of the other
// threads of the barrier) to the cluster's threads that acquire the arrivals' phase.
__device__ __forceinline__ void fence_acq_rel_cluster()
{
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// One poll of a phase of this CTA's mbarrier, with acquire at cluster scope (for phases completed
// by arrivals from other CTAs of the cluster); the sleeping form suspends up to `hint_ns`.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(hint_ns)
                 : "memory");
    return ok != 0;
}

// Generic-proxy accesses of global memory ordered with this thread's async-proxy accesses (bulk
// copies) of global memory.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from global memory into
// this CTA's shared memory, completion counted on this CTA's mbarrier.
__device__ __forceinline__ void bulk_load_global(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    if (!smem_ok(dst, bytes) || !smem_ok(bar, 8)) return;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Every thread of every CTA of the cluster arrives, then waits for all (release / acquire at
// cluster scope).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Polls of a cluster-scope wait: each suspends for at most CLUSTER_WAIT_HINT_NS (the thread also
// wakes when the phase completes); together they give up after a second or more.
constexpr uint32_t CLUSTER_WAIT_HINT_NS = 1000;
constexpr int CLUSTER_WAIT_LIMIT = 1 << 21;

// Bounded wait on a phase of this CTA's mbarrier (acquire at cluster scope). Like wait_bar, it
// gives up after CLUSTER_WAIT_LIMIT polls (flagging DEVERR_TIMEOUT and this CTA's abort flag) or
// as soon as this CTA gave up.
__device__ __noinline__ bool wait_cluster_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
#pragma unroll 1
    for (int i = 0; i < CLUSTER_WAIT_LIMIT; ++i) {
        if (mbar_try_wait_cluster(bar, parity, CLUSTER_WAIT_HINT_NS)) return true;
        if (*abort_flag) return false;
    }
    atomicOr(&g_dev_error, DEVERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait_cluster(bar, parity, 0)) return true;
    return wait_cluster_slow(bar, parity, abort_flag);
}

}  // namespace kda
