// Asynchronous global -> shared copies (cp.async, 16 bytes, L2 only), used
// by the HBM-bound kernels to keep loads in flight without holding
// registers.  Groups are per thread: a thread that reads back only what it
// copied needs no barrier, just cp_async_wait.
#pragma once

#include <cstdint>

namespace awq {

// src_bytes < 16 zero-fills the rest of the 16 bytes (0: all zeros, src unread).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes = 16) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's copy groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace awq
