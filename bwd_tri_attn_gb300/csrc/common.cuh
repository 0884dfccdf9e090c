// Shared device helpers for the triangle-attention kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tri_attn.h"

namespace triattn {

// Problem description passed by value to every kernel. node: 0 = starting node (pair tensors
// [B,S,N,H,d]: slices along pair axis 1), 1 = ending node (pair tensors [B,N,S,H,d]: slices
// along pair axis 2).
struct Dims {
  int B, S, N, H, d;
  float scale;
  int node;
};

// Row index of position n of slice (b, i) in the [rows, H*d] view of a pair tensor of the given
// node (kernels pass it as a compile-time constant).
__host__ __device__ inline int64_t pos_row(const Dims &g, int b, int i, int n, int node) {
  return (int64_t)b * g.S * g.N + (node ? (int64_t)n * g.S + i : (int64_t)i * g.N + n);
}


__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(((uint32_t)v) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&h);
}

// 2^x on the multi-function unit (PTX ex2.approx; relative error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (three-input max.f32 of sm_100-family GPUs).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// How the backward spreads its work: NC clusters (one per resident cluster slot of the device),
// and KMAX dBias partial slots per head in the workspace.
struct BwdSplit {
  int NC, KMAX;
};

// ---------------------------------------------------------------- power-of-two operand scaling
// The tensor-core operands that meet an FP16 factor (P, dS) must be FP16 themselves, and FP16
// covers only magnitudes 2^-14 .. 65504 at full precision, while BF16 inputs span 2^-126 .. 2^127.
// Each (batch, slice, head) block of V (forward) and of Q, K, V, dO (backward) is therefore
// multiplied by 2^s before the BF16 -> FP16 conversion, s chosen from the block's largest exponent
// so that its largest magnitude lands in [2^T, 2^(T+1)); the accumulators are multiplied by the
// inverse power of two on the way out. Both multiplications are exact, so the results are the
// unscaled arithmetic's, bit for bit, wherever that arithmetic stays in FP16's normal range.
// Blocks whose largest magnitude M lies in [2^-40, 2^41) get the exact target binade; outside it the
// exponent of the nearest bound is used. Scale exponents then lie in [T - 40, T + 40] (|s| <= 54),
// so each single factor and each product of two is a normal FP32 value; products of three are
// applied as two multiplications.
constexpr int kScaleExpLimit = 40;
constexpr int kTargetQK = 14;       // Q, K (backward) and V (forward): largest magnitude in [2^14, 2^15)
// Backward V and dO: their scale factors multiply into the scale of dS' = P (dP' - w D), whose
// magnitude is below d * 2^(tv + to + 3) (|dP|, |D| <= d max|dO| max|V|); tv + to = 11 - log2(d)
// keeps it below 2^14, well inside FP16.
template <int HD>
struct BwdTargets {
  static constexpr int TV = 3, TO = HD == 32 ? 3 : 4;
  static_assert(TV + TO + 3 + (HD == 32 ? 5 : 4) <= 14, "dS' bound");
};

// Scale exponent for a block whose largest BF16 exponent field is e (0: the block is zero or
// subnormal and keeps scale 1).
__host__ __device__ inline int scale_exp(int e, int target) {
  if (e == 0) return 0;
  int m = e - 127;  // floor(log2 M)
  m = m < -kScaleExpLimit ? -kScaleExpLimit : (m > kScaleExpLimit ? kScaleExpLimit : m);
  return target - m;
}

// 2^n as an FP32 value, n in [-126, 127].
__device__ __forceinline__ float exp2i(int n) { return __int_as_float((n + 127) << 23); }

// Running maximum of the BF16 exponent fields held in the two halves of a packed pair
// (call bf16x2_exp_final on the accumulated word).
__device__ __forceinline__ uint32_t bf16x2_exp_max(uint32_t acc, uint32_t w) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w & 0x7f807f80u));
  return r;
}
__device__ __forceinline__ int bf16x2_exp_final(uint32_t acc) {
  const uint32_t lo = acc & 0xffffu, hi = acc >> 16;
  return (int)((lo > hi ? lo : hi) >> 7);
}

// Running maximum of the BF16 exponent fields of the eight values in a 16-byte chunk.
__device__ __forceinline__ uint32_t exp_max4(uint32_t acc, const uint4 &v) {
  return bf16x2_exp_max(bf16x2_exp_max(bf16x2_exp_max(bf16x2_exp_max(acc, v.x), v.y), v.z), v.w);
}

// Maximum of v over the CTA (NT threads, a multiple of 32); every thread gets the result.
// red: NT / 32 ints of shared memory.
template <int NT>
__device__ __forceinline__ int block_max(int v, int *red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int m = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) m = max(m, red[w]);
  __syncthreads();
  return m;
}

// 16-byte streaming load (read once: no L1 allocation).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}


// Device status codes written by bounded waits (host reads them lazily).
constexpr int kStatusTimeout = 1;

}  // namespace triattn
