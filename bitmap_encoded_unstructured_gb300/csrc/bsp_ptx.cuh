// Inline-PTX helpers for sm_100-family asynchronous copies and barriers:
// mbarrier (init / expect-tx / bounded try-wait) and the 1-D bulk copy
// engine (cp.async.bulk, global -> shared, completion counted in bytes on
// an mbarrier).  No multicast anywhere.
#pragma once

#include <cstdint>

namespace bspx {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One arrival that also raises the expected transaction count by `bytes`.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Spin cap of every device-side wait: past it the wait gives up, the
// kernel records BSP_ERR_TIMEOUT in the handle's error word and returns.
constexpr uint32_t kSpinCap = 1u << 22;

// Wait for phase `parity` of `bar`; false if `cap` polls ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t cap = kSpinCap)
{
    for (uint32_t i = 0; i < cap; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// One poll that may suspend the thread for up to `hint_ns` nanoseconds; the
// thread resumes as soon as the phase completes, so a waiting warp takes
// no issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// mbar_wait_bounded with suspending polls: at most `cap` polls of at most
// `hint_ns` each.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t cap,
                                                uint32_t hint_ns = 1000)
{
    for (uint32_t i = 0; i < cap; ++i)
        if (mbar_try_wait_sleep(bar, parity, hint_ns)) return true;
    return false;
}

// ---- thread-block clusters (the prefill kernel's split-K pairs)

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives (release) and waits
// (acquire).  The .aligned forms need the whole warp to execute them
// together, and the compiler does not reconverge a warp before inline asm:
// a warp that comes from a per-lane polling loop (bounded mbarrier waits)
// may still be split, and its parts would then arrive in different phases
// of the barrier.  __syncwarp() reconverges it first.
__device__ __forceinline__ void cluster_sync()
{
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-window address, in the CTA of cluster rank `rank`, of this CTA's
// shared-memory address `saddr` (the same offset).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// 16-byte store to a cluster shared-window address (another CTA's memory).
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

// Bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace bspx
