// kvx_async.cuh -- cp.async (global -> shared, 16 bytes, asynchronous)
// wrappers for the streaming kernels (kvx_diag.cu, kvx_ridge.cu): each thread
// copies its own words into a shared-memory ring and waits for its own
// groups, so loads in flight hold no registers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace {

// cp.async of 16 bytes global -> shared, bypassing L1; src_bytes = 0 writes
// zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src,
                                           uint32_t src_bytes) {
  const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(gmem_src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace
