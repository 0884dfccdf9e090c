// Host-side launch helpers: per-device, thread-safe one-time set-up records.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace triattn {

constexpr int kMaxDevices = 64;

// The current device, refused when it is outside the range the per-device records cover.
inline cudaError_t current_device(int *dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  return (*dev < 0 || *dev >= kMaxDevices) ? cudaErrorInvalidDevice : cudaSuccess;
}

// One bit per device: set once a kernel's set-up (its shared-memory attribute, which the runtime
// keeps per device, and the register check) has succeeded there. Host threads may race to run
// the set-up; it is idempotent, so the only cost of a race is doing it twice.
struct DeviceOnce {
  std::atomic<uint64_t> bits{0};
  bool done(int dev) const { return (bits.load(std::memory_order_acquire) >> dev) & 1u; }
  void mark(int dev) { bits.fetch_or(uint64_t{1} << dev, std::memory_order_release); }
};

// A per-device integer computed once (0 = not yet known).
struct DeviceValue {
  std::atomic<int> v[kMaxDevices] = {};
  int get(int dev) const { return v[dev].load(std::memory_order_acquire); }
  void set(int dev, int x) { v[dev].store(x, std::memory_order_release); }
};

}  // namespace triattn
