// Host helper: the one-time opt-in of a kernel to more than 48 KB of dynamic shared memory, per
// device.  The first launch on each device sets the attribute; concurrent first calls from several
// host threads are serialised by a mutex, later calls only read an atomic flag.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace qv {

struct SmemOptIn {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  std::atomic<bool> done[kMaxDevices] = {};

  template <typename Kernel>
  cudaError_t ensure(Kernel kern, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e != cudaSuccess) return e;
      done[dev].store(true, std::memory_order_release);
    }
    return cudaSuccess;
  }
};

}  // namespace qv
