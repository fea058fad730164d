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

}  // namespace ccv
