// Host side of the kernel launches: per-device launch settings shared by every
// host thread. A launch site keeps one LaunchMemo and reads or updates it under
// its mutex only; the launch itself happens outside the lock. A kernel's
// dynamic shared-memory limit is only ever raised, so a concurrent launch never
// sees it lowered.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include <mutex>

namespace specv {

constexpr int kMaxDevices = 64;

struct LaunchMemo {
  std::mutex mu;
  size_t granted[kMaxDevices] = {};    // dynamic shared memory granted so far
  size_t grid_smem[kMaxDevices] = {};  // shared-memory size `grid` was computed for
  int grid[kMaxDevices] = {};
};

// The current device, or -1 when it cannot be read or is out of range.
static inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Caller holds m.mu: raise `kern`'s dynamic shared-memory limit on `dev` to `smem`.
static inline bool grant_smem_locked(LaunchMemo& m, const void* kern, int dev, size_t smem) {
  if (smem <= m.granted[dev]) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return false;
  m.granted[dev] = smem;
  return true;
}

}  // namespace specv
