// Test-only library: exercises the attention kernels' bounded-wait machinery
// (sync.cuh) on a real GPU without faulting or hanging it.
//
// One CTA, two warps. Warp 0 waits on an mbarrier that nothing ever arrives
// on; after the wait limit it must raise the CTA's abort flag and the status
// word and return false. Warp 1 waits on a second such mbarrier and must leave
// through the abort flag raised by warp 0 (or, at the latest, through its own
// limit). Both record whether their wait succeeded and how long it took, and
// the kernel then returns normally: the context stays usable.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sync.cuh"

using namespace triattn;
using namespace triattn::sm100;

namespace {

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(int *status, int *ok_out, unsigned long long *ns_out) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ volatile int flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const Abort ab{&flag, status};
  const uint64_t t0 = globaltimer_ns();
  // warp 1 starts its wait a little later, so that warp 0's limit expires first
  if (warp == 1) {
    while (globaltimer_ns() - t0 < 100000000ull) {
    }
  }
  const bool ok = wait_bar_warp(smem_u32(&bars[warp]), 0, ab);
  const uint64_t t1 = globaltimer_ns();
  if (lane == 0) {
    ok_out[warp] = ok ? 1 : 0;
    ns_out[warp] = (unsigned long long)(t1 - t0);
  }
}

}  // namespace

// Runs the probe on the current device and waits for it. status, ok_out (2 ints) and
// ns_out (2 u64) are device pointers. Returns the CUDA error code of launch + sync.
extern "C" int wait_timeout_probe(int *status, int *ok_out, unsigned long long *ns_out) {
  wait_timeout_kernel<<<1, 64>>>(status, ok_out, ns_out);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return (int)e;
}

// The wait limit the kernels use, in nanoseconds.
extern "C" unsigned long long wait_limit_ns() { return kWaitLimitNs; }
