// Host-side TMA tensor-map construction for the pair tensors and the pair bias.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace triattn {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// TMA view of a BF16 pair tensor. Starting node ([B,S,N,H,d] in memory): 4-D (d, H, N, B*S),
// batch and slice merged. Ending node ([B,N,S,H,d]): 5-D (d, H, S, N, B), dimensions in order of
// increasing stride. One TMA box is `rows` consecutive positions of one (b, slice, head): `rows`
// x d elements, swizzled to the operand layout (SW64 for d = 32: 64-byte rows; SW32 for
// d = 16). Positions past N read as zeros (and are not written by stores). Kernels address it
// through load_rows / store_rows below.
inline cudaError_t make_rows_map(CUtensorMap *m, const void *ptr, const Dims &g, int rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t row = 2ull * g.d * g.H;  // bytes of one (b, slice, position) row
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5] = {1, 1, 1, 1, 1};
  cuuint32_t rank;
  if (!g.node) {
    rank = 4;
    const cuuint64_t d4[4] = {(cuuint64_t)g.d, (cuuint64_t)g.H, (cuuint64_t)g.N, (cuuint64_t)g.B * g.S};
    const cuuint64_t s4[3] = {2ull * g.d, row, row * g.N};
    const cuuint32_t b4[4] = {(cuuint32_t)g.d, 1, (cuuint32_t)rows, 1};
    for (int k = 0; k < 4; ++k) dims[k] = d4[k], box[k] = b4[k];
    for (int k = 0; k < 3; ++k) strides[k] = s4[k];
  } else {
    rank = 5;
    const cuuint64_t d5[5] = {(cuuint64_t)g.d, (cuuint64_t)g.H, (cuuint64_t)g.S, (cuuint64_t)g.N, (cuuint64_t)g.B};
    const cuuint64_t s5[4] = {2ull * g.d, row, row * g.S, row * g.S * g.N};
    const cuuint32_t b5[5] = {(cuuint32_t)g.d, 1, 1, (cuuint32_t)rows, 1};
    for (int k = 0; k < 5; ++k) dims[k] = d5[k], box[k] = b5[k];
    for (int k = 0; k < 4; ++k) strides[k] = s5[k];
  }
  const CUtensorMapSwizzle sw = g.d == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D view (j, k, b*H + h) of a BF16 [B*H, NP, NP] square matrix stack with
// NP a multiple of 128; one box is 64 columns x 128 rows, 128-byte swizzled.
inline cudaError_t make_square_map(CUtensorMap *m, const void *ptr, int NP, int BH) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)NP, (cuuint64_t)NP, (cuuint64_t)BH};
  cuuint64_t strides[2] = {2ull * NP, 2ull * NP * NP};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D view (k, j, b*H + h) of the BF16 pair bias [B*H, N, N] (N a multiple of 8, so
// that rows start on 16-byte boundaries); one box is 64 keys x 128 query rows,
// 128-byte swizzled. Rows and keys past N read as zeros.
inline cudaError_t make_bias_map(CUtensorMap *m, const void *ptr, int N, int BH) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {2ull * N, 2ull * N * N};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace triattn
