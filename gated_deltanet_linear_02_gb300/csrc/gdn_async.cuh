// gdn_async.cuh -- sm_100-family asynchronous-copy and barrier primitives as
// inline PTX: mbarriers, 1-D TMA bulk copies, and bounded waits.
//
// Every wait in libgdn is bounded. A wait that exceeds its limit returns
// false. The caller then records GDN_ERR_TIMEOUT in its device error word and
// leaves the kernel cleanly, instead of spinning forever.
#pragma once

#include <stdint.h>

namespace gdn {

// A wait gives up after this many nanoseconds (2 s): longer than any
// legitimate memory latency, short enough that a broken pipeline ends.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Ends an mbarrier's life, so that its word may be initialised again.
__device__ __forceinline__ void mbar_inval(uint32_t bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (TMA) and the cluster.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// The dynamic shared-memory block rounded up to a 128-byte boundary. It is
// formed as an offset into the __shared__ array itself, so the compiler still
// knows the pointer addresses shared memory. That lets it move shared loads
// past global stores, which may not alias them.
__device__ __forceinline__ unsigned char *smem_aligned128(unsigned char *raw)
{
    return raw + ((128u - (smem_u32(raw) & 127u)) & 127u);
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA / tensor core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 1-D bulk copy global -> shared through the TMA unit; completion is counted in
// bytes on `bar`. Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// 1-D bulk copy shared -> global through the TMA unit, added to this thread's
// current bulk group. Both addresses 16-byte aligned, bytes a multiple of 16.
// The issuing thread fences (fence_proxy_async_smem) after the shared writes,
// and waits for its groups (bulk_wait_read / bulk_wait_all) before the shared
// memory is reused or the CTA exits.
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// This thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// One try that may suspend the thread for up to `hint_ns` nanoseconds while the
// phase is still open: the warp sleeps instead of spinning, so it takes no
// issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

// mbar_wait_bounded with suspending tries (see mbar_try_wait_sleep), for
// kernels where most warps wait most of the time.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}

// Waits for phase `parity` of `bar` to complete, for at most WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u && global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}

// ---- programmatic dependent launch
// A kernel launched with the programmatic-stream-serialization attribute may
// start before the kernel ahead of it in the stream has finished. It must call
// grid_dep_wait() before touching memory that kernel writes (or reads and it
// overwrites): the wait returns once that kernel has completed and its memory
// operations are visible. In a kernel launched without the attribute it
// returns at once. grid_dep_launch() lets the kernel behind this one start
// early; it only changes scheduling, never what the waiting kernel sees.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- thread-block clusters and distributed shared memory

// The shared::cluster address of the shared-memory location `addr` in the CTA
// of rank `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t cluster_addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(cluster_addr) : "memory");
    return v;
}

// Barrier over every thread of every CTA in the cluster, with release /
// acquire ordering of their memory accesses. Each thread of the cluster must
// reach it.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

}  // namespace gdn
