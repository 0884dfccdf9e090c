// Softmax-backward correction D (HBM-bound streaming kernel).
//
// D[b,i,h,j] = sum_c dO[b,i,j,h,c] * (O[b,i,j,h,c] + Ores[b,i,j,h,c]) in FP32.
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract): computing this correction
// from the BF16-rounded forward output loses precision; adding back the
// stored BF16 approximation of the output-rounding residual recovers the FP32
// output to within BF16-of-a-residual, so D is formed in FP32 from O + Ores.
// With Ores == NULL the kernel uses O alone (the uncompensated variant).
//
// Work split: every thread loads one 16-byte chunk (8 BF16) of each of dO, O
// and Ores, so a warp reads 512 contiguous bytes of each tensor. The d/8
// chunks of one (position, head) sit in neighbouring lanes and are combined
// with a fixed xor-shuffle tree, so the summation order is fixed.
#include "common.cuh"

namespace triattn {

constexpr int kDPosPerBlock = 32;
constexpr int kDThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

template <int HD, bool kResidual>
__global__ void __launch_bounds__(kDThreads)
bwd_d_kernel(Dims g, const uint4 *__restrict__ dO, const uint4 *__restrict__ O,
             const uint4 *__restrict__ Ores, float *__restrict__ Dout, int64_t positions) {
  extern __shared__ float sD[];  // [kDPosPerBlock][H]
  constexpr int cph = HD / 8;    // 16-byte chunks per (position, head)
  const int cpp = g.H * cph;     // chunks per position
  const int64_t p0 = (int64_t)blockIdx.x * kDPosPerBlock;
  const int total = kDPosPerBlock * cpp;  // a multiple of 64: warps stay converged
  for (int c = threadIdx.x; c < total; c += kDThreads) {
    const int64_t p = p0 + c / cpp;
    float acc = 0.f;
    if (p < positions) {
      const int64_t idx = p * cpp + (c % cpp);
      const uint4 a = ld_stream(dO + idx);
      const uint4 o = ld_stream(O + idx);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w};
      const uint32_t ov[4] = {o.x, o.y, o.z, o.w};
      if (kResidual) {
        const uint4 r = ld_stream(Ores + idx);
        const uint32_t rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = bf2_to_f2(av[e]), fo = bf2_to_f2(ov[e]), fr = bf2_to_f2(rv[e]);
          acc = fmaf(fa.x, fo.x + fr.x, acc);
          acc = fmaf(fa.y, fo.y + fr.y, acc);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = bf2_to_f2(av[e]), fo = bf2_to_f2(ov[e]);
          acc = fmaf(fa.x, fo.x, acc);
          acc = fmaf(fa.y, fo.y, acc);
        }
      }
    }
#pragma unroll
    for (int off = 1; off < cph; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if ((c % cph) == 0) sD[(c / cpp) * g.H + (c % cpp) / cph] = acc;
  }
  __syncthreads();
  for (int t = threadIdx.x; t < kDPosPerBlock * g.H; t += kDThreads) {
    const int pl = t % kDPosPerBlock, h = t / kDPosPerBlock;
    const int64_t p = p0 + pl;
    if (p < positions) {
      // memory row p -> (b * S + slice i) and position j; the ending node stores slices innermost
      int64_t bi, j;
      if (!g.node) {
        bi = p / g.N;
        j = p % g.N;
      } else {
        const int64_t sn = (int64_t)g.S * g.N, b = p / sn, r = p % sn;
        bi = b * g.S + r % g.S;
        j = r / g.S;
      }
      Dout[(bi * g.H + h) * g.N + j] = sD[pl * g.H + h];
    }
  }
}

cudaError_t launch_bwd_d(const Dims &g, const uint16_t *dO, const uint16_t *O, const uint16_t *Ores,
                         float *Dout, cudaStream_t stream) {
  const int64_t positions = (int64_t)g.B * g.S * g.N;
  const unsigned blocks = (unsigned)((positions + kDPosPerBlock - 1) / kDPosPerBlock);
  const size_t smem = sizeof(float) * kDPosPerBlock * g.H;
  auto *a = reinterpret_cast<const uint4 *>(dO);
  auto *o = reinterpret_cast<const uint4 *>(O);
  auto *r = reinterpret_cast<const uint4 *>(Ores);
  if (g.d == 32) {
    if (Ores) bwd_d_kernel<32, true><<<blocks, kDThreads, smem, stream>>>(g, a, o, r, Dout, positions);
    else bwd_d_kernel<32, false><<<blocks, kDThreads, smem, stream>>>(g, a, o, r, Dout, positions);
  } else {
    if (Ores) bwd_d_kernel<16, true><<<blocks, kDThreads, smem, stream>>>(g, a, o, r, Dout, positions);
    else bwd_d_kernel<16, false><<<blocks, kDThreads, smem, stream>>>(g, a, o, r, Dout, positions);
  }
  return cudaGetLastError();
}

}  // namespace triattn
