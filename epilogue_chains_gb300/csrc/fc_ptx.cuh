// fc_ptx.cuh -- inline-PTX building blocks for sm_103a: mbarriers with bounded waits.
// (TMA and tcgen05 wrappers live in fc_tc.cuh.)
#pragma once

#include <stdint.h>

namespace fc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Suspend-time hint of one try_wait, in ns: a waiting thread is parked by the hardware until the
// phase completes or this much time has passed, instead of spinning and taking issue slots from
// the warps that do the work.
constexpr uint32_t kTryWaitHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kTryWaitHintNs)
        : "memory");
    return ok != 0;
}

// Default budget of one bounded wait, in SM clock cycles (~1 s at 2 GHz).
constexpr long long kWaitBudget = 2000000000LL;
// A wait reads the watchdog flag (a global-memory load) only once it has lasted this many cycles
// (~0.5 ms): a normal pipeline wait ends within microseconds and never pays for the load, which
// would otherwise delay its noticing the phase change by a memory round trip.
constexpr long long kFlagPollAfter = 1LL << 20;

// Wait for phase `parity` of an mbarrier to complete, for at most `budget` SM cycles.  On expiry
// (or when another thread already raised the watchdog flag) the flag is set and false is
// returned; the caller must then unwind without issuing new asynchronous work.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int* flag,
                                                  long long budget = kWaitBudget) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (++spins % 8u == 0u) {
            const long long dt = clock64() - t0;
            if (dt > kFlagPollAfter && *reinterpret_cast<volatile int*>(flag) != 0) return false;
            if (dt > budget) {
                atomicExch(flag, 1);
                return false;
            }
        }
    }
    return true;
}

// Global-memory flags between CTAs of one grid (all co-resident): a release store after the
// writer's data, an acquire load before the reader's.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Wait until *p == want, for at most `budget` SM cycles (then the watchdog flag is set and false
// returned, as for mbar_wait_bounded).  Spins on the load: the waits it serves last microseconds,
// below the wake-up granularity of a sleep.
__device__ __forceinline__ bool flag_wait_bounded(const int* p, int want, int* flag,
                                                  long long budget = kWaitBudget) {
    if (ld_acquire_gpu(p) == want) return true;
    const long long t0 = clock64();
    uint32_t spins = 0;
    while (ld_relaxed_gpu(p) != want) {
        if (++spins % 8u != 0u) continue;
        const long long dt = clock64() - t0;
        if (dt > kFlagPollAfter && *reinterpret_cast<volatile int*>(flag) != 0) return false;
        if (dt > budget) {
            atomicExch(flag, 1);
            return false;
        }
    }
    fence_acq_rel_gpu();   // with the relaxed load that saw `want`: an acquire of the writer's release
    return true;
}

// Drain wait after a failure: the copies or MMAs this CTA already issued must land before its
// shared memory and TMEM are released, whatever other CTAs reported, so the watchdog flag is not
// consulted; only the time budget bounds the wait.  Returns false if it ran out.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity,
                                                long long budget = kWaitBudget / 8) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (++spins % 8u == 0u && clock64() - t0 > budget) return false;
    }
    return true;
}

}  // namespace fc
