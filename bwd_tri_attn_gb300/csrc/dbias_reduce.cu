// Fixed-order reduction of the per-slice-group dBias partials (HBM-bound).
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract): the bias is shared by all
// slices, so dBias is a reduction over slices; it is done with ordered partial
// sums rather than floating-point atomics. The backward kernel leaves one FP32
// partial per slice group g in the workspace; this kernel adds the G partials
// in the order g = 0, 1, ..., G-1 and rounds once to BF16.
//
// Partial layout: [G][B*H][N][N] FP32, element (j, k) at j*N + k.
#include "common.cuh"

namespace triattn {

constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads)
dbias_reduce_kernel(const float *__restrict__ partial, int G, int64_t elems,
                    uint16_t *__restrict__ dBias) {
  const int64_t e0 = ((int64_t)blockIdx.x * kReduceThreads + threadIdx.x) * 4;
  if (e0 >= elems) return;
  if (e0 + 4 <= elems && (elems % 4) == 0) {
    float4 acc = *reinterpret_cast<const float4 *>(partial + e0);
    for (int gi = 1; gi < G; ++gi) {
      const float4 v = __ldcs(reinterpret_cast<const float4 *>(partial + (int64_t)gi * elems + e0));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const uint2 out = make_uint2((uint32_t)f32_to_bf16_rn(acc.x) | ((uint32_t)f32_to_bf16_rn(acc.y) << 16),
                                 (uint32_t)f32_to_bf16_rn(acc.z) | ((uint32_t)f32_to_bf16_rn(acc.w) << 16));
    *reinterpret_cast<uint2 *>(dBias + e0) = out;
  } else {
    for (int64_t e = e0; e < e0 + 4 && e < elems; ++e) {
      float acc = partial[e];
      for (int gi = 1; gi < G; ++gi) acc += partial[(int64_t)gi * elems + e];
      dBias[e] = f32_to_bf16_rn(acc);
    }
  }
}

cudaError_t launch_dbias_reduce(const float *partial, int G, int64_t elems, uint16_t *dBias,
                                cudaStream_t stream) {
  const int64_t threads = (elems + 3) / 4;
  const unsigned blocks = (unsigned)((threads + kReduceThreads - 1) / kReduceThreads);
  dbias_reduce_kernel<<<blocks, kReduceThreads, 0, stream>>>(partial, G, elems, dBias);
  return cudaGetLastError();
}

}  // namespace triattn
