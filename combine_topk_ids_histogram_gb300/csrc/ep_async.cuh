// Bulk asynchronous shared -> global copies (cp.async.bulk) and the proxy fence they need.
#pragma once
#include <cstdint>

namespace ep {

// Shared-memory bytes written by ordinary stores must be ordered before the copy engine reads
// them: every writer runs fence_proxy_async_smem(), then a barrier, then the copies are issued.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from shared to global memory.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, unsigned bytes) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(ssrc));
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gdst), "r"(s), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's copies have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's copies have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace ep
