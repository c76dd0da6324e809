// Split programmatic-dependent-launch controls and bulk asynchronous shared -> global copies,
// for kernels that do work before waiting on the previous kernel in the stream.
#pragma once
#include <cstdint>

namespace ep {

// Wait until every earlier kernel in the stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel in the stream start launching (its own wait still orders its reads).
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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
