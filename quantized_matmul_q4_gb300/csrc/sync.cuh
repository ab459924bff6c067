// mbarrier / bulk-copy helpers with bounded waits (sm_103a).
#pragma once

#include <cstdint>

namespace q4mm {

// Set when a bounded wait gives up; read by q4mm_device_status().
__device__ __forceinline__ void flag_timeout(int *status) {
    if (status) atomicOr(status, 1);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread for up to `hint_ns`
// nanoseconds while the phase is incomplete, so waiting warps do not spin.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Suspend-time hint of the bounded wait, in nanoseconds (0: no hint, the
// hardware's own try_wait time limit).
#ifndef Q4MM_WAIT_HINT_NS
#define Q4MM_WAIT_HINT_NS 20000
#endif

// Wait for phase `parity` of `bar` to complete, giving up after about
// `limit_cycles` SM cycles.  Returns false on time-out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long limit_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
#if Q4MM_WAIT_HINT_NS > 0
    while (!mbar_try_wait_sleep(bar, parity, Q4MM_WAIT_HINT_NS)) {
#else
    while (!mbar_try_wait(bar, parity)) {
#endif
        if (clock64() - t0 > limit_cycles) return false;
    }
    return true;
}

// As mbar_wait_bounded, but also gives up (returns false) once *abort is set
// by another thread of the CTA that has already given up.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t *bar, uint32_t parity, long long limit_cycles,
                                                    const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 2000)) return true;
        if (*abort || clock64() - t0 > limit_cycles) return false;
    }
}

// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_wait_abortable, by spinning on non-blocking tests: for a single
// thread whose next instructions must follow the phase's completion at
// once (a tensor-core issuer, whose idle time is idle tensor pipe).
__device__ __forceinline__ bool mbar_spin_abortable(uint64_t *bar, uint32_t parity, long long limit_cycles,
                                                    const volatile int *abort) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_test_wait(bar, parity)) return true;
        if (*abort || clock64() - t0 > limit_cycles) return false;
    }
}

// 1-D bulk copy global → shared, completion counted on `bar` in bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Prefetch `bytes` (a multiple of 16, 16-byte aligned address) into L2.
// A hint only: no data is returned, so it is safe before the wait on the
// previous kernel even for memory that kernel writes.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// Orders this thread's earlier shared-memory accesses (and those it has
// acquired from other threads) before later async-proxy operations on shared
// memory, such as a bulk copy into a buffer that was just read.
__device__ __forceinline__ void fence_async_proxy() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// About one second at GB300 clocks: far beyond any legitimate wait here.
// (Launches take their limit as a parameter; this is its value unless a
// test asks for a shorter one.)
constexpr long long kWaitLimitCycles = 2000000000LL;

}  // namespace q4mm
