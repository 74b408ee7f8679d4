// pa_ptx.cuh -- inline-PTX helpers for sm_103a: mbarriers, 1-D bulk async
// copies (TMA) into shared memory, programmatic dependent launch, bounded
// waits.  Device code only; no state.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pa {

// A bounded wait gives up after this long (ns of %globaltimer) or this many
// polls, whichever comes first, and reports PA_ERRBIT_TIMEOUT.  The wait
// for a CTA's own copies and tensor-core work still in flight, before it
// leaves, has the same limits in every build (kDrainLimit*).
constexpr uint64_t kDrainLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kDrainLimitPolls = 1u << 28;
#ifdef PA_TEST_WAIT_POLLS
// Test build: every other wait polls without blocking (mbarrier.test_wait)
// and gives up after PA_TEST_WAIT_POLLS polls, so it runs out on an ordinary
// call and the give-up path can be checked on the GPU.
constexpr uint64_t kWaitLimitNs = kDrainLimitNs;
constexpr uint32_t kWaitLimitPolls = PA_TEST_WAIT_POLLS;
constexpr bool kShortWaits = true;
#else
constexpr uint64_t kWaitLimitNs = kDrainLimitNs;
constexpr uint32_t kWaitLimitPolls = kDrainLimitPolls;
constexpr bool kShortWaits = false;
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy and other threads.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if the
// wait gave up (time or poll limit) or *abort became non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if constexpr (kShortWaits) {
        for (uint32_t polls = 0; polls < kWaitLimitPolls; ++polls)
            if (mbar_test_wait(bar, parity)) return true;
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t polls = 1; polls < kWaitLimitPolls; ++polls) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((polls & 31u) == 0u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
    return false;
}

// The wait for a CTA's own copies or tensor-core work in flight before it
// leaves: `never` is a flag nothing sets, and the limits are the full ones
// in every build (in the ordinary build this is exactly mbar_wait).
__device__ __forceinline__ bool mbar_drain_wait(uint64_t *bar, uint32_t parity,
                                                volatile int *never) {
    if constexpr (kShortWaits) {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t polls = 1; polls < kDrainLimitPolls; ++polls) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((polls & 31u) == 0u && globaltimer_ns() - t0 > kDrainLimitNs) return false;
        }
        return false;
    } else {
        return mbar_wait(bar, parity, never);
    }
}

// L2 policy for data read once (the K/V stream).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_nohint(void *dst, const void *src, uint32_t bytes,
                                                uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled bulk copy (TMA) through a tensor map; x is the innermost
// coordinate (elements) and must satisfy the same 16-byte rule.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int x, int y, int z,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 4-D tiled bulk copy (TMA) through a tensor map; same rules as tma_load_3d.
__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, int x, int y, int z,
                                            int w, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                        uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Programmatic dependent launch: wait for the preceding grid's completion and
// memory flush / allow the next grid to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Hardware base-2 exponential (MUFU), flushes denormals; ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace pa
