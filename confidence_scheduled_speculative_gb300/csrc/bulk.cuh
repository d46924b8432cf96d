// bulk.cuh -- helpers for TMA bulk copies (cp.async.bulk) completing on
// shared-memory mbarriers (used by the scatter).
#pragma once

#include <cstdint>

namespace dspark {

constexpr unsigned long long kWaitLimitNs = 200000000ull;  // 200 ms: the default limit

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Wait for the given phase parity of an mbarrier: a non-blocking test in a
// loop, given up (false) once limit_ns of wall time have passed since the
// first test; limit_ns = 0 tests once.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    const unsigned long long start = global_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (global_ns() - start >= limit_ns) return false;
        __nanosleep(32);
    }
}

// Announce `bytes` of transaction on the barrier (with this thread's arrival)
// and start a bulk copy of `bytes` from global `src` to shared `dst` that
// completes them.  dst, src and bytes are multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

}  // namespace dspark
