// Unit probe of the tcgen05 / TMA building blocks (test-only library).
//
// One CTA, 128 threads. Checks, against host matmuls, the three operand
// layouts the attention kernels rely on:
//   S  = A * B^T           A, B: [128 x d] BF16, K-major, TMA-swizzled (SW64 for d=32, SW32 for d=16)
//   O  = P * V             P: FP16 in TMEM (A operand from TMEM), V: [128 x d] FP16 MN-major (TMA-swizzled)
//   O2 = X^T * V           X: FP16 [128 x 128] written by threads into a SW128 MN-major shared tile
// where P = X = fp16(S * xscale). Results go to S_out [128][128], O_out, O2_out [128][d] (FP32).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm100.cuh"

using namespace triattn::sm100;

namespace {

// Bounded wait (1 s): on expiry sets *err and returns false; the probe then skips to teardown.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, int *err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 1000000000ull) {
      atomicExch(err, 1);
      return false;
    }
  }
  return true;
}

struct __align__(1024) ProbeSmem {
  uint16_t A[128 * 32];
  uint16_t B[128 * 32];
  uint16_t V[128 * 32];
  uint16_t X[128 * 128];  // SW128 MN-major: [8-row group][M half][8 rows][128 B]
  uint64_t bar_tma, bar_mma;
  uint32_t tmem_base;
};

template <int HD>
__global__ void __launch_bounds__(128) probe_kernel(const __grid_constant__ CUtensorMap mA,
                                                    const __grid_constant__ CUtensorMap mB,
                                                    const __grid_constant__ CUtensorMap mV, float xscale,
                                                    float *S_out, float *O_out, float *O2_out, int *err) {
  extern __shared__ __align__(1024) uint8_t raw[];
  ProbeSmem &sm = *reinterpret_cast<ProbeSmem *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid / 32;
  const uint32_t bar_tma = smem_u32(&sm.bar_tma), bar_mma = smem_u32(&sm.bar_mma);
  constexpr uint32_t ROWB = HD * 2;  // bytes per operand row
  constexpr uint32_t SW = HD == 32 ? kSwizzle64B : kSwizzle32B;
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_tma, 3 * 128 * ROWB);
    tma_load_4d(smem_u32(sm.A), &mA, bar_tma, 0, 0, 0, 0);
    tma_load_4d(smem_u32(sm.B), &mB, bar_tma, 0, 0, 0, 0);
    tma_load_4d(smem_u32(sm.V), &mV, bar_tma, 0, 0, 0, 0);
  }
  bool ok = wait_bounded(bar_tma, 0, err);
  // S = A B^T: K-major both, K-steps of 16 elements = 32 bytes inside each swizzled row
  if (tid == 0 && ok) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_f16(128, 128, true, true, false, false);
    for (int ks = 0; ks < HD / 16; ++ks) {
      const uint64_t da = smem_desc(smem_u32(sm.A) + ks * 32, 16, 8 * ROWB, SW);
      const uint64_t db = smem_desc(smem_u32(sm.B) + ks * 32, 16, 8 * ROWB, SW);
      mma_ss(tbase, da, db, idesc, ks > 0);
    }
    mma_commit(bar_mma);
  }
  // V -> FP16 in place (layout unchanged)
  {
    uint32_t *v = reinterpret_cast<uint32_t *>(sm.V);
    for (int e = tid; e < 128 * HD / 2; e += 128) v[e] = bf16x2_to_f16x2(v[e]);
  }
  ok = __syncthreads_and(ok);
  if (ok) ok = wait_bounded(bar_mma, 0, err);
  tc_fence_after();
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  float s[128];
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(tbase + lane_off + c * 32, r);
    tmem_wait_ld(r);
    for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[e]);
  }
  for (int e = 0; e < 128; ++e) S_out[tid * 128 + e] = s[e];
  // P = fp16(S*xscale) packed two per column into TMEM columns [0, 64)
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    for (int e = 0; e < 32; ++e) r[e] = pack_f16x2(s[c * 64 + 2 * e] * xscale, s[c * 64 + 2 * e + 1] * xscale);
    tmem_st32(tbase + lane_off + c * 32, r);
  }
  tmem_wait_st();
  // X (same values) into the SW128 MN-major tile: row = tid (K index), 128 columns (M index)
  {
    const uint32_t base = smem_u32(sm.X);
    for (int half = 0; half < 2; ++half)
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t w[4];
        for (int e = 0; e < 4; ++e) {
          const int col = half * 64 + ch * 8 + 2 * e;
          w[e] = pack_f16x2(s[col] * xscale, s[col + 1] * xscale);
        }
        const uint32_t addr = base + (tid / 8) * 2048 + half * 1024 + (tid % 8) * 128 + ((ch ^ (tid % 8)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                     "r"(w[3])
                     : "memory");
      }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  ok = __syncthreads_and(ok);
  if (tid == 0 && ok) {
    tc_fence_after();
    // O = P V: A from TMEM (8 columns per 16-key step), B = V MN-major (N = HD contiguous)
    constexpr uint32_t idesc_pv = idesc_f16(128, HD, false, false, false, true);
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t dv = smem_desc(smem_u32(sm.V) + ks * 16 * ROWB, 16, 8 * ROWB, SW);
      mma_ts(tbase + 128, tbase + ks * 8, dv, idesc_pv, ks > 0);
    }
    // O2 = X^T V: A = X^T from SMEM, MN-major SW128 (M halves 1 KB apart = LBO, 8-row K groups 2 KB apart = SBO)
    constexpr uint32_t idesc_x = idesc_f16(128, HD, false, false, true, true);
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t dx = smem_desc(smem_u32(sm.X) + ks * 4096, 1024, 2048, kSwizzle128B);
      const uint64_t dv = smem_desc(smem_u32(sm.V) + ks * 16 * ROWB, 16, 8 * ROWB, SW);
      mma_ss(tbase + 128 + 64, dx, dv, idesc_x, ks > 0);
    }
    mma_commit(bar_mma);
  }
  if (ok) ok = wait_bounded(bar_mma, 1, err);
  tc_fence_after();
  {
    uint32_t r[32];
    tmem_ld32(tbase + lane_off + 128, r);
    tmem_wait_ld(r);
    for (int e = 0; e < HD; ++e) O_out[tid * HD + e] = __uint_as_float(r[e]);
    tmem_ld32(tbase + lane_off + 128 + 64, r);
    tmem_wait_ld(r);
    for (int e = 0; e < HD; ++e) O2_out[tid * HD + e] = __uint_as_float(r[e]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int make_map(CUtensorMap *m, const void *ptr, int hd) {
  cuuint64_t dims[4] = {(cuuint64_t)hd, 1, 128, 1};
  cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)hd * 2, (cuuint64_t)hd * 2 * 128};
  cuuint32_t box[4] = {(cuuint32_t)hd, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  auto fn = encode_fn();
  if (!fn) return -1;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, hd == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

}  // namespace

extern "C" int tcgen05_probe(const void *A, const void *B, const void *V, int hd, float xscale, float *S_out,
                             float *O_out, float *O2_out, int *err) {
  if (hd != 16 && hd != 32) return -3;
  CUtensorMap mA, mB, mV;
  if (make_map(&mA, A, hd) || make_map(&mB, B, hd) || make_map(&mV, V, hd)) return -1;
  const size_t smem = sizeof(ProbeSmem) + 1024;
  if (hd == 32) {
    cudaFuncSetAttribute(probe_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    probe_kernel<32><<<1, 128, smem>>>(mA, mB, mV, xscale, S_out, O_out, O2_out, err);
  } else {
    cudaFuncSetAttribute(probe_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    probe_kernel<16><<<1, 128, smem>>>(mA, mB, mV, xscale, S_out, O_out, O2_out, err);
  }
  if (cudaGetLastError() != cudaSuccess) return -4;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : -5;
}
