// Bounded waits for the warp-specialised kernels.
//
// Every spin on an mbarrier has a time limit. When it expires the waiting
// thread raises the CTA's shared abort flag and the library's device status
// word, and returns false; every other wait in the CTA then sees the abort flag
// and returns false at once, so all roles fall through to teardown instead of
// hanging. The host reads the status word with tri_attn_device_status().
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace triattn {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: normal waits last microseconds

struct Abort {
  volatile int *flag;  // shared memory, one per CTA
  int *status;         // global device status word
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Abort &ab) {
  if (sm100::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = sm100::globaltimer_ns();
  while (true) {
    if (sm100::mbar_try_wait(bar, parity)) return true;
    if (*ab.flag) return false;
    if (sm100::globaltimer_ns() - t0 > kWaitLimitNs) {
      *ab.flag = 1;
      atomicExch(ab.status, kStatusTimeout);
      return false;
    }
  }
}

// As wait_bar, with acquire at cluster scope (for barriers that peer CTAs arrive on).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, const Abort &ab) {
  if (sm100::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = sm100::globaltimer_ns();
  while (true) {
    if (sm100::mbar_try_wait_cluster(bar, parity)) return true;
    if (*ab.flag) return false;
    if (sm100::globaltimer_ns() - t0 > kWaitLimitNs) {
      *ab.flag = 1;
      atomicExch(ab.status, kStatusTimeout);
      return false;
    }
  }
}

// Waits on an mbarrier with every lane of the warp; true only if all lanes succeeded.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Abort &ab) {
  const bool ok = wait_bar(bar, parity, ab);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait used at teardown: ignores the abort flag (it only drains work in flight).
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = sm100::globaltimer_ns();
  while (!sm100::mbar_try_wait(bar, parity))
    if (sm100::globaltimer_ns() - t0 > kWaitLimitNs) break;
}

}  // namespace triattn
