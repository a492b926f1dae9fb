// qk_ptx.cuh -- thin inline-PTX wrappers for sm_103a: shared-memory
// mbarriers, bulk async copies (global -> shared), bounded waits.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace qk {

// Device status bits (the word lives in qk_api.cu; kernels get its address).
enum : unsigned { STATUS_TIMEOUT = 1u };

// Spin budget of one bounded mbarrier wait.  try_wait already suspends the
// thread for a hardware-chosen interval per attempt, so this bound is far
// beyond any legitimate wait (a bulk copy completes in microseconds).
constexpr uint32_t kWaitSpins = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// A wait gives up after this long (time, checked every 256 polls) or after
// kWaitSpins polls, whichever comes first.
constexpr uint64_t kWaitNs = 2000000000ull;

// Bounded wait for phase `parity` of `bar` to complete.  Returns false when
// the budget runs out, after setting STATUS_TIMEOUT in *status.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned* status,
                                                  uint64_t limit_ns = kWaitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < kWaitSpins; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
    }
    atomicOr(status, STATUS_TIMEOUT);
    return false;
}

// try_wait that lets the hardware suspend the thread for up to `ns`
// nanoseconds while the phase is incomplete (it resumes when the phase
// completes), for long waits by threads that should not spin.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait with suspension between checks (same time bound).
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t* bar, uint32_t parity, unsigned* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < (1u << 24); ++i) {
        if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
        if (globaltimer_ns() - t0 > kWaitNs) break;
    }
    atomicOr(status, STATUS_TIMEOUT);
    return false;
}

// Bounded wait that also gives up when another warp of the CTA has already
// given up (*abort set); on its own timeout it sets *abort and the status.
// Between checks the warp is suspended by the hardware until the phase
// completes (or a microsecond passes), so waiting warps take no issue slots
// from the working ones.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t* bar, uint32_t parity, unsigned* status,
                                                    volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1; i < (1u << 24); ++i) {
        if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitNs) break;
    }
    *abort = 1;
    atomicOr(status, STATUS_TIMEOUT);
    return false;
}

// Evict-first L2 policy for data streamed exactly once (weights of a GEMV).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Evict-last L2 policy for small data many CTAs read (prepped activations).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from
// global to this CTA's shared memory, completing on `bar` (complete_tx).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 16-byte asynchronous global -> shared copy (per thread, no register
// staging), grouped with commit / wait_group.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// 16-byte cp.async to a shared address given as a 32-bit offset, with an L2
// cache policy (e.g. evict-first for bytes read once); issued only when
// off < lim (unsigned).
__device__ __forceinline__ void cp_async16_if_lt(uint32_t sdst, const void* src, uint64_t policy, uint32_t off,
                                                 uint32_t lim) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.lt.u32 q, %3, %4;\n\t"
        "@q cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;\n\t}" ::"r"(sdst),
        "l"(src), "l"(policy), "r"(off), "r"(lim)
        : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's memory to be visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace qk
