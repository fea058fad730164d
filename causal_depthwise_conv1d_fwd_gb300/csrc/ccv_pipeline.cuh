// Shared-memory staging primitives: per-thread asynchronous global -> shared
// copies (cp.async) with commit / wait groups.  A thread only ever waits for
// its own copies, so no wait here depends on another thread or block.
#pragma once

#include <cstdint>

namespace ccv {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Per-thread asynchronous 16-byte copy global -> shared (L1 bypassed), and
// the commit / wait-group pair that tracks this thread's copies.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Bring the line holding p into L1 (no register result, no wait).  Only for
// data that no thread writes during the launch.
__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Wait until at most n of this thread's copy groups are pending (n <= 0:
// all done; n >= 7: at most 7).  In a fully unrolled loop n folds to a
// constant and only one wait instruction remains.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
    switch (n) {
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        default:
            if (n >= 7) cp_async_wait<7>();
            else cp_async_wait<0>();
    }
}

}  // namespace ccv
