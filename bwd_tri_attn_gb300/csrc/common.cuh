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

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// How the backward spreads its work: NC clusters (one per resident cluster slot of the device),
// and KMAX dBias partial slots per head in the workspace.
struct BwdSplit {
  int NC, KMAX;
};

// Device status codes written by bounded waits (host reads them lazily).
constexpr int kStatusTimeout = 1;

}  // namespace triattn
