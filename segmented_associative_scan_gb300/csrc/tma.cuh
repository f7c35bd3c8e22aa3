// TMA bulk copies and mbarriers (inline PTX, sm_90+ / sm_103a) for the streaming kernel.
//
// Only the untiled, non-multicast form is used: cp.async.bulk global -> shared of this
// CTA, completing on an mbarrier with a transaction byte count. Source and destination
// must be 16-byte aligned and the size a multiple of 16 bytes; the launcher only picks
// the streaming kernel when every copy it will issue satisfies that.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rlca {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy (the TMA unit).
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also announces `bytes` of incoming transactions.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

// Bounded wait for the phase with the given parity to complete. Each try_wait may
// suspend the thread for a hardware-defined interval; after `limit` failed tries the
// wait gives up and returns false (the caller marks its outputs invalid).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int limit)
{
    const uint32_t addr = smem_addr(bar);
    for (int i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy `bytes` (multiple of 16) from global `src` to this CTA's shared `dst`, both
// 16-byte aligned; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

}  // namespace rlca
