// Asynchronous-copy pipeline helpers: shared-memory mbarriers, bulk (TMA)
// global -> shared copies that complete on an mbarrier, and a bounded wait.
//
// Every wait on an mbarrier in this library goes through mbar_wait_bounded:
// after `limit_ns` nanoseconds of the global timer without the phase
// completing it records the cause in the library's device error word (read
// back by tq_device_errors) and returns false, so that the kernel can drain
// and return instead of spinning.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace tqk {

// bits of the device error word
constexpr uint32_t kErrScanWait = 1u;      // a scan tile's copy did not complete in time
constexpr uint32_t kErrSelfTestWait = 2u;  // the bounded-wait self-test ran out (expected)
constexpr uint32_t kErrQuantWait = 4u;     // a quantize CTA's operand fragments did not land in time

// a copy from HBM lands within microseconds; one second means it never will
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

// make mbarrier initialisation visible to the async proxy (bulk copies)
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// order this thread's earlier generic-proxy shared accesses before later
// async-proxy accesses (a buffer read by the warp is refilled by a bulk copy)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// one arrival that also announces `bytes` of transactions for this phase
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// plain arrival (no transactions)
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, completing on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended for up to hint_ns while
// the phase is incomplete (it resumes when the phase completes), so a waiting
// warp does not spin through issue slots other warps need.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// one suspension of a bounded wait: far below the limit, far above a copy's latency
constexpr uint32_t kWaitSuspendNs = 20000u;

// Waits for the phase with the given parity to complete, at most `limit_ns`.
// On time-out sets `code` in *err (if err is not null) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns, uint32_t* err,
                                                  uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait_suspend(bar, parity, kWaitSuspendNs)) {
        if (global_ns() - t0 > limit_ns) {
            if (err) atomicOr(err, code);
            return false;
        }
    }
    return true;
}

}  // namespace tqk
