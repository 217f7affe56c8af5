// Opt-in to more than 48 KB of dynamic shared memory, per device.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>

namespace moe {

constexpr int kMaxDevices = 64;

// A kernel's dynamic shared memory limit (cudaFuncAttributeMaxDynamicSharedMemorySize)
// is an attribute of the kernel on one device.  `done` keeps, per device
// ordinal, the largest value already set for the kernel; a call asking for
// no more returns without a driver call.  Safe to call from several host
// threads (a lost race sets the same attribute twice).
inline cudaError_t opt_in_smem(const void* kernel, std::atomic<size_t> (&done)[kMaxDevices],
                               size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && bytes <= done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e != cudaSuccess || !cached) return e;
  size_t cur = done[dev].load(std::memory_order_relaxed);
  while (cur < bytes &&
         !done[dev].compare_exchange_weak(cur, bytes, std::memory_order_release,
                                          std::memory_order_relaxed)) {
  }
  return cudaSuccess;
}

}  // namespace moe
