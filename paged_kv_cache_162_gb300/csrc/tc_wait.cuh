// Bounded mbarrier waits and tcgen05 fences shared by the tensor-core
// prefix kernel (prefix_tc.cuh, inside decode.cu) and the runtime's
// self-test of their give-up path (runtime.cu).  A wait polls
// mbarrier.try_wait at most `limit` times and reports failure instead of
// spinning on: a kernel that gives up sets PKV_DEVERR_TIMEOUT, frees what it
// holds and returns, so no wait can hang the device.
#ifndef PKV_TC_WAIT_CUH
#define PKV_TC_WAIT_CUH

#include <cstdint>

constexpr long long kTcWaitLimit = 1ll << 20;  // try_wait rounds before giving up

__device__ __forceinline__ void tc_mbar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool tc_mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait for phase `parity`; false after `limit` rounds or as soon
// as another role has given up (*abort set)
__device__ __forceinline__ bool tc_mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                             long long limit = kTcWaitLimit) {
    for (long long i = 0; i < limit; ++i) {
        if (tc_mbar_try(bar, parity)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    return false;
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
#endif  // PKV_TC_WAIT_CUH
