// Triangle-attention block around the attention core: LayerNorm, the q/k/v, pair-bias and gate
// projections, the attention (fwd.cu, bwd.cu), the sigmoid gate and the output projection,
// forward and backward.
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract, first sentence) places the attention in
// AlphaFold3-style models without describing the layers around it; this is the plainest reading
// of that model family's triangle-attention layer (include/tri_module.h states it in full).
//
// Forward (M = B N^2 pair positions, hd = H d):
//   mod_ln_fwd_kernel     z -> zt (BF16), mean, 1/std; pair bias zt . wb (transposed for the ending node)
//   GEMM                  zt W^T -> q | k | v | gl (one product, the epilogue routes each 32-column
//                         chunk to its tensor)
//   attention             tri_attn forward on q, k, v, bias, mask
//   mod_gate_kernel       go = sigmoid(gl) O
//   GEMM                  go Wo^T -> out
// Backward:
//   GEMM + gate epilogue  dgo = dout Wo; the epilogue writes dO = dgo s and dgl = dgo O s (1 - s)
//                         (s = sigmoid(gl)): dgo never reaches memory
//   GEMM (split over M)   dWo partials = dout^T go, then a fixed-order sum over the splits
//   attention             tri_attn backward -> dq, dk, dv, dbias
//   GEMM                  dzt = [dq | dk | dv | dgl] W (FP32), the four tensors read as one K-segmented operand
//   mod_ln_bwd_kernel     dzt + dbias wb -> dz; per-CTA partial sums of dgamma, dbeta, dwb
//   GEMM (split over M)   dW partials = [dq | dk | dv | dgl]^T zt, then a fixed-order sum
//
// The GEMM is one persistent tcgen05 kernel for every product: M = 128 x N = 128 or 256 tiles (the
// narrower for products at most 128 wide), K steps of 64 through a TMA ring, two TMEM
// accumulators so that one tile's epilogue overlaps the next tile's main loop, BF16 and FP32
// outputs leaving through TMA stores. Operands are K-major (row-major [rows][K]) or MN-major (the
// transposed operand mode, [K][rows]); one operand may be split into up to four tensors along K
// (K-major) or M (MN-major), so [dq | dk | dv | dgl] is read where the attention left it. Products
// summed over the pair positions split K into fixed chunks of rows; each chunk's FP32 partial is
// written out and the partials are added in a fixed order, so every weight gradient is the same
// bits on every call.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "launch.cuh"
#include "plan.cuh"
#include "sm100.cuh"
#include "sync.cuh"
#include "tmap.cuh"
#include "tri_module.h"

namespace triattn {
using namespace sm100;

int *device_status_word();

namespace {

// sigmoid in FP32 from the fast exponential and reciprocal (a few FP32 ulp plus about one per
// unit of |x|; 0 below x = -87)
__device__ __forceinline__ float sigm(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float lo_bf(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ================================================================ GEMM
enum { kOutBF16 = 0, kOutF32 = 1, kOutGate = 2 };

struct MGemmArgs {
  int M, N, K, Kc, T;     // D[t][m][n] = sum over k in [t Kc, min(K, t Kc + Kc)) of A(m, k) B(n, k)
  int segA, nsegA;        // A's tensors hold segA elements each along K (K-major A) or M (MN-major A)
  void *D0, *D1, *D2, *D3;  // kOutBF16: column segments of segD columns, row stride segD; kOutF32: [T][M][N]
  int segD;               // (the outputs' tensor maps are built from these at plan time)
  const uint16_t *P, *G;  // kOutGate: [M][N] attention output and gate logits
  uint16_t *dP, *dG;      // kOutGate: [M][N] their gradients
};

template <int BN_, int kOut_>
struct MGemmCfg {
  static constexpr int BM = 128, BN = BN_, BK = 64;
  // BF16 and FP32 outputs leave through TMA stores of 32 x 32 pieces staged per warp (two pieces,
  // 64- or 128-byte rows, swizzled like the store's tensor map); the gate epilogue transposes
  // through a padded 32 x 33 FP32 tile instead
  static constexpr bool TMA_OUT = kOut_ != 2;
  static constexpr int PIECE = 32 * 32 * (kOut_ == 1 ? 4 : 2);
  static constexpr int NST = BN == 256 ? (kOut_ == 1 ? 3 : 4) : (kOut_ == 0 ? 6 : 5);
  static constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE = A_BYTES + B_BYTES;
  static constexpr int MN_BOX = BK * 128;  // one 64-wide MN-major box: BK rows of 128 bytes
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_CPW = BN / 32 / (EPI_WARPS / 4);  // 32-column chunks per epilogue warp
  static constexpr int EPI_PITCH = 33;
  static constexpr int EPI_TILE = TMA_OUT ? 2 * PIECE : 32 * EPI_PITCH * 4;
  static constexpr int OFF_EPI = NST * STAGE;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_TILE;
  static constexpr int B_FULL = 0, B_EMPTY = NST, B_ACCF = 2 * NST, B_ACCE = B_ACCF + 2, B_DONE = B_ACCE + 2,
                       NBAR = B_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 64 + 32 * EPI_WARPS;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(BN == 128 || BN == 256, "tile width");
  static_assert(STAGE % 1024 == 0 && A_BYTES % 1024 == 0 && OFF_EPI % 1024 == 0, "1 KB alignment (swizzle atoms)");
  static_assert(EPI_TILE % 1024 == 0 || !TMA_OUT, "staging pieces on 1 KB boundaries");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// The gate epilogue's 8 consecutive values v = dgo of row m, columns n .. n + 7, with the attention
// output pv and gate logits gv there: dP = dgo s and dG = dgo O s (1 - s), s = sigmoid(gl).
__device__ __forceinline__ void gate_store8(const MGemmArgs &a, int m, int n, const float (&v)[8], const uint4 &pv,
                                            const uint4 &gv) {
  const int64_t off = (int64_t)m * a.N + n;
  const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
  uint32_t od[4], og[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const float d0 = v[2 * x], d1 = v[2 * x + 1];
    const float s0 = sigm(lo_bf(gw[x])), s1 = sigm(hi_bf(gw[x]));
    od[x] = pack_bf16x2(d0 * s0, d1 * s1);
    og[x] = pack_bf16x2(d0 * lo_bf(pw[x]) * (s0 * (1.f - s0)), d1 * hi_bf(pw[x]) * (s1 * (1.f - s1)));
  }
  *reinterpret_cast<uint4 *>(a.dP + off) = make_uint4(od[0], od[1], od[2], od[3]);
  *reinterpret_cast<uint4 *>(a.dG + off) = make_uint4(og[0], og[1], og[2], og[3]);
}

template <bool kAMN, bool kBMN, int kOut, int BN>
__global__ void __launch_bounds__(MGemmCfg<BN, kOut>::NTHREADS, 1)
    mod_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                    const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mA3,
                    const __grid_constant__ CUtensorMap mB, const __grid_constant__ CUtensorMap mO0,
                    const __grid_constant__ CUtensorMap mO1, const __grid_constant__ CUtensorMap mO2,
                    const __grid_constant__ CUtensorMap mO3, const MGemmArgs a, int *status) {
  using C = MGemmCfg<BN, kOut>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int k) { return sb0 + C::OFF_BAR + 8u * (uint32_t)k; };
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_MISC);
  const Abort ab{reinterpret_cast<volatile int *>(misc + 1), status};
  const int mt = (a.M + C::BM - 1) / C::BM, nt = (a.N + C::BN - 1) / C::BN;
  const int ntiles = a.T * mt * nt;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_FULL + s), 1);
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_ACCF + s), 1);
      mbar_init(bar(C::B_ACCE + s), 32 * C::EPI_WARPS);
    }
    mbar_init(bar(C::B_DONE), 1);
    misc[1] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sb0 + C::OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = misc[0];
  auto tile_of = [&](int u, int &t, int &m0, int &n0) {
    t = u / (mt * nt);
    const int r = u - t * (mt * nt);
    m0 = (r / nt) * C::BM;
    n0 = (r % nt) * C::BN;
  };
  // K blocks of split t (at least one: the host picks T = ceil(K / Kc))
  auto kblocks = [&](int t, int &k0) {
    k0 = t * a.Kc;
    return (min(a.K, k0 + a.Kc) - k0 + C::BK - 1) / C::BK;
  };
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    bool ok = true;
    int it = 0;
    if (lane == 0) {
      tma_prefetch_map(&mA0);
      tma_prefetch_map(&mB);
    }
    for (int u = blockIdx.x; u < ntiles && ok; u += gridDim.x) {
      int t, m0, n0, kbeg;
      tile_of(u, t, m0, n0);
      const int nk = kblocks(t, kbeg);
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int st = it % C::NST;
        if (it >= C::NST) ok = wait_bar_warp(bar(C::B_EMPTY + st), ((it / C::NST) - 1) & 1, ab);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t dst = sb0 + st * C::STAGE, fb = bar(C::B_FULL + st);
          const int k0 = kbeg + kb * C::BK;
          mbar_arrive_expect_tx(fb, C::STAGE);
          if constexpr (kAMN) {
#pragma unroll
            for (int x = 0; x < C::BM / 64; ++x) {
              const int mm = m0 + 64 * x, s = min(mm / a.segA, a.nsegA - 1);
              const CUtensorMap *pa = s == 0 ? &mA0 : s == 1 ? &mA1 : s == 2 ? &mA2 : &mA3;
              tma_load_3d(dst + x * C::MN_BOX, pa, fb, mm - s * a.segA, k0, 0);
            }
          } else {
            const int s = min(k0 / a.segA, a.nsegA - 1);
            const CUtensorMap *pa = s == 0 ? &mA0 : s == 1 ? &mA1 : s == 2 ? &mA2 : &mA3;
            tma_load_3d(dst, pa, fb, k0 - s * a.segA, m0, 0);
          }
          if constexpr (kBMN) {
#pragma unroll
            for (int x = 0; x < C::BN / 64; ++x) tma_load_3d(dst + C::A_BYTES + x * C::MN_BOX, &mB, fb, n0 + 64 * x, k0, 0);
          } else {
            tma_load_3d(dst + C::A_BYTES, &mB, fb, k0, n0, 0);
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0)  // let the copies in flight land before the CTA exits
      for (int x = max(0, it - C::NST); x < it; ++x) drain_bar(bar(C::B_FULL + x % C::NST), (x / C::NST) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp, elect.sync)
    constexpr uint32_t idesc = idesc_f16(C::BM, C::BN, true, true, kAMN, kBMN);
    constexpr uint64_t a_step = kAMN ? (16 * 128) >> 4 : 32 >> 4;
    constexpr uint64_t b_step = kBMN ? (16 * 128) >> 4 : 32 >> 4;
    bool ok = true;
    int it = 0, tl = 0;
    for (int u = blockIdx.x; u < ntiles && ok; u += gridDim.x, ++tl) {
      int t, m0, n0, kbeg;
      tile_of(u, t, m0, n0);
      const int nk = kblocks(t, kbeg);
      const int acc = tl & 1;
      if (tl >= 2) ok = wait_bar_warp(bar(C::B_ACCE + acc), ((tl >> 1) - 1) & 1, ab);
      if (!ok) break;
      tc_fence_after();
      const uint32_t dacc = tb + acc * C::BN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int st = it % C::NST;
        ok = wait_bar_warp(bar(C::B_FULL + st), (it / C::NST) & 1, ab);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = sb0 + st * C::STAGE, sbb = sa + C::A_BYTES;
        const uint64_t da = kAMN ? smem_desc(sa, C::MN_BOX, 1024, kSwizzle128B) : smem_desc(sa, 16, 1024, kSwizzle128B);
        const uint64_t db =
            kBMN ? smem_desc(sbb, C::MN_BOX, 1024, kSwizzle128B) : smem_desc(sbb, 16, 1024, kSwizzle128B);
#pragma unroll
        for (int ks = 0; ks < C::BK / 16; ++ks)
          mma_ss_e(dacc, da + a_step * ks, db + b_step * ks, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
        mma_commit_e(bar(C::B_EMPTY + st));
      }
      if (!ok) break;
      mma_commit_e(bar(C::B_ACCF + acc));
    }
    mma_commit_e(bar(C::B_DONE));
    if (lane == 0) drain_bar(bar(C::B_DONE), 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue: TMEM -> registers -> global
    // Each warp reads its chunks (EPI_CPW x 32 columns of its TMEM lane quarter, thread = row) into
    // registers and hands the accumulator back before its last stores, so the next tile's MMAs
    // overlap them. BF16 and FP32 outputs: the thread writes its row of a chunk into a staging piece
    // in the store map's swizzle and one lane issues a TMA store of the 32 x 32 piece (two pieces
    // per warp in turn). Gate epilogue: the rows go through a padded transpose tile, so that each
    // thread holds 8 consecutive values of four rows for its loads of O and gl and its stores.
    const int q = warp & 3;
    const int cbase = ((warp - 2) >> 2) * (32 * C::EPI_CPW);
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    const uint32_t stg_s = sb0 + C::OFF_EPI + (warp - 2) * C::EPI_TILE;
    float *stg = reinterpret_cast<float *>(sm + C::OFF_EPI + (warp - 2) * C::EPI_TILE);
    const int rq = lane >> 2, cq = lane & 3;
    int tl = 0, pc = 0;  // tiles, staged pieces of this warp
    for (int u = blockIdx.x; u < ntiles; u += gridDim.x, ++tl) {
      int t, m0, n0;
      tile_of(u, t, m0, n0);
      const int acc = tl & 1;
      const int mrow = m0 + q * 32 + rq;
      const bool rows_live = m0 + q * 32 < a.M;  // (warp-uniform) this warp's 32 rows reach into the product
      // Chunks are read in groups of GRP (all of them, or two at a time where the registers of
      // four would spill); the accumulator goes back to the MMA warp once the last group is in
      // registers.
      constexpr int GRP = (C::EPI_CPW > 2 && kOut != kOutBF16) ? 2 : C::EPI_CPW;
      bool ok = true;
#pragma unroll
      for (int g0 = 0; g0 < C::EPI_CPW; g0 += GRP) {
        // the gate epilogue's inputs at this thread's store positions, requested before the waits
        uint4 pv[GRP][4], gv[GRP][4];
        if constexpr (kOut == kOutGate) {
#pragma unroll
          for (int k = 0; k < GRP; ++k) {
            const int col = n0 + cbase + 32 * (g0 + k) + 8 * cq;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (mrow + 8 * i < a.M && col < a.N) {
                const int64_t off = (int64_t)(mrow + 8 * i) * a.N + col;
                pv[k][i] = *reinterpret_cast<const uint4 *>(a.P + off);
                gv[k][i] = *reinterpret_cast<const uint4 *>(a.G + off);
              }
          }
        }
        if (g0 == 0) {
          ok = wait_bar_warp(bar(C::B_ACCF + acc), (tl >> 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
        }
        uint32_t r[GRP][32];
#pragma unroll
        for (int k = 0; k < GRP; ++k)
          if (n0 + cbase + 32 * (g0 + k) < a.N) tmem_ld32(tb + lrow + acc * C::BN + cbase + 32 * (g0 + k), r[k]);
        tmem_wait_ld(r);
        if (g0 + GRP >= C::EPI_CPW) {
          tc_fence_before();
          mbar_arrive(bar(C::B_ACCE + acc));
        }
#pragma unroll
        for (int k = 0; k < GRP; ++k) {
          const int n = n0 + cbase + 32 * (g0 + k);
          if (n >= a.N || !rows_live) break;  // uniform across the warp
          if constexpr (C::TMA_OUT) {
            const uint32_t piece = stg_s + (uint32_t)(pc & 1) * C::PIECE;
            if (pc >= 2) {  // the store issued from this piece two pieces ago has read it
              if (lane == 0) bulk_wait_group_read<1>();
              __syncwarp();
            }
            if constexpr (kOut == kOutBF16) {
              // row = lane: 64 bytes, 16-byte chunk c at c ^ ((row / 2) mod 4) (64-byte swizzle)
#pragma unroll
              for (int c = 0; c < 4; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(piece + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)),
                             "r"(pack_bf16x2(__uint_as_float(r[k][8 * c]), __uint_as_float(r[k][8 * c + 1]))),
                             "r"(pack_bf16x2(__uint_as_float(r[k][8 * c + 2]), __uint_as_float(r[k][8 * c + 3]))),
                             "r"(pack_bf16x2(__uint_as_float(r[k][8 * c + 4]), __uint_as_float(r[k][8 * c + 5]))),
                             "r"(pack_bf16x2(__uint_as_float(r[k][8 * c + 6]), __uint_as_float(r[k][8 * c + 7])))
                             : "memory");
            } else {
              // row = lane: 128 bytes, 16-byte chunk c at c ^ (row mod 8) (128-byte swizzle)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(piece + lane * 128 + ((c ^ (lane & 7)) << 4)),
                             "r"(r[k][4 * c]), "r"(r[k][4 * c + 1]), "r"(r[k][4 * c + 2]), "r"(r[k][4 * c + 3])
                             : "memory");
            }
            fence_proxy_async_smem();  // the generic-proxy writes before the async-proxy read
            __syncwarp();
            if (lane == 0) {
              if constexpr (kOut == kOutBF16) {
                const int sg = n / a.segD;
                const CUtensorMap *mo = sg == 0 ? &mO0 : sg == 1 ? &mO1 : sg == 2 ? &mO2 : &mO3;
                tma_store_3d(mo, piece, n - sg * a.segD, m0 + q * 32, 0);
              } else {
                tma_store_3d(&mO0, piece, n, m0 + q * 32, t);
              }
              bulk_commit_group();
            }
            ++pc;
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) stg[lane * C::EPI_PITCH + j] = __uint_as_float(r[k][j]);
            __syncwarp();
            const int col = n + 8 * cq;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float v[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = stg[(rq + 8 * i) * C::EPI_PITCH + 8 * cq + j];
              if (mrow + 8 * i < a.M && col < a.N) gate_store8(a, mrow + 8 * i, col, v, pv[k][i], gv[k][i]);
            }
            __syncwarp();
          }
        }
      }
      if (!ok) break;
    }
    if constexpr (C::TMA_OUT) {
      if (lane == 0) bulk_wait_group<0>();  // every store has been performed before the CTA exits
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, C::TMEM_COLS);
  }
}

// 2-D TMA view (inner, outer) of a BF16 row-major matrix with `pitch` elements per row, as a 3-D
// map with one batch; one box is 64 inner elements (128 bytes, 128-byte swizzled) x `rows`.
// Elements past the extents read as zeros.
cudaError_t make_mat_map(CUtensorMap *m, const void *ptr, int64_t inner, int64_t outer, int64_t pitch, int rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, 1};
  cuuint64_t strides[2] = {(cuuint64_t)(2 * pitch), (cuuint64_t)(2 * pitch * outer)};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D TMA view (inner, outer, batch) of a row-major output for 32 x 32 stores: BF16 with 64-byte
// box rows (64-byte swizzle) or FP32 with 128-byte box rows (128-byte swizzle). Rows past `outer`
// within a batch are not written.
cudaError_t make_out_map(CUtensorMap *m, void *ptr, bool f32, int64_t inner, int64_t outer, int64_t batch) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const int64_t es_bytes = f32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)(es_bytes * inner), (cuuint64_t)(es_bytes * inner * outer)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// One planned product. A(m, k): K-major A is row-major [M][K] (split along K into the given
// tensors of segA columns each), MN-major A is row-major [K][M] (split along M into tensors of
// segA columns each); B(n, k): K-major [N][K] or MN-major [K][N].
template <bool kAMN, bool kBMN, int kOut, int BN>
struct MGemmT {
  using C = MGemmCfg<BN, kOut>;
  CUtensorMap mA[4], mB, mO[4];
  MGemmArgs a;
  int grid;
  // io: the outputs (kOutBF16: D0..D3 and segD; kOutF32: D0; kOutGate: P, G, dP, dG)
  cudaError_t plan(const uint16_t *const *A, int nA, int segA, const uint16_t *B, int M, int N, int K, int Kc,
                   const MGemmArgs &io) {
    cudaError_t e = cudaSuccess;
    for (int s = 0; s < 4 && e == cudaSuccess; ++s) {
      const uint16_t *p = A[s < nA ? s : 0];
      e = kAMN ? make_mat_map(&mA[s], p, segA, K, segA, C::BK) : make_mat_map(&mA[s], p, segA, M, segA, C::BM);
    }
    if (e == cudaSuccess) e = kBMN ? make_mat_map(&mB, B, N, K, N, C::BK) : make_mat_map(&mB, B, K, N, K, C::BN);
    a = io;
    a.M = M;
    a.N = N;
    a.K = K;
    a.Kc = Kc;
    a.T = (K + Kc - 1) / Kc;
    a.segA = segA;
    a.nsegA = nA;
    void *d[4] = {io.D0, io.D1, io.D2, io.D3};
    for (int s = 0; s < 4 && e == cudaSuccess; ++s) {
      if (kOut == kOutBF16) {
        const int nseg = (N + io.segD - 1) / io.segD;
        e = make_out_map(&mO[s], d[s < nseg ? s : 0], false, io.segD, M, 1);
      } else if (kOut == kOutF32) {
        e = make_out_map(&mO[s], d[0], true, N, M, a.T);
      } else {
        mO[s] = mB;  // (unused by the gate epilogue)
      }
    }
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    e = current_device(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    static DeviceOnce ready;
    if (!ready.done(dev)) {
      e = cudaFuncSetAttribute(mod_gemm_kernel<kAMN, kBMN, kOut, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_ALLOC);
      if (e != cudaSuccess) return e;
      ready.mark(dev);
    }
    const int64_t tiles = (int64_t)a.T * ((M + C::BM - 1) / C::BM) * ((N + C::BN - 1) / C::BN);
    grid = (int)std::min<int64_t>(tiles, nsm);
    return cudaSuccess;
  }
  cudaError_t launch(int *status, cudaStream_t st) const {
    mod_gemm_kernel<kAMN, kBMN, kOut, BN><<<grid, C::NTHREADS, C::SMEM_ALLOC, st>>>(
        mA[0], mA[1], mA[2], mA[3], mB, mO[0], mO[1], mO[2], mO[3], a, status);
    return cudaGetLastError();
  }
};

// The tile width follows the product's width: N <= 128 takes 128-column tiles (no MMA work or
// epilogue warps spent on empty columns), wider products 256-column tiles.
template <bool kAMN, bool kBMN, int kOut>
struct MGemm {
  MGemmT<kAMN, kBMN, kOut, 128> narrow;
  MGemmT<kAMN, kBMN, kOut, 256> wide;
  bool use_narrow = false;
  cudaError_t plan(const uint16_t *const *A, int nA, int segA, const uint16_t *B, int M, int N, int K, int Kc,
                   const MGemmArgs &io) {
    use_narrow = N <= 128;
    return use_narrow ? narrow.plan(A, nA, segA, B, M, N, K, Kc, io) : wide.plan(A, nA, segA, B, M, N, K, Kc, io);
  }
  cudaError_t launch(int *status, cudaStream_t st) const {
    return use_narrow ? narrow.launch(status, st) : wide.launch(status, st);
  }
};

MGemmArgs out_bf16(void *d0, void *d1, void *d2, void *d3, int seg) {
  MGemmArgs o{};
  o.D0 = d0;
  o.D1 = d1;
  o.D2 = d2;
  o.D3 = d3;
  o.segD = seg;
  return o;
}

// ================================================================ LayerNorm and pair bias
// CC / 8 lanes per pair position, 8 consecutive channels (16 bytes) per lane, 32 / (CC / 8)
// positions per warp at a time; sums over a position's channels by a fixed xor-shuffle tree
// within its lane group. The bias of head h is the dot product of the BF16-rounded zt row (the
// values the projections read) with wb[h], written by lane h of the group.
template <int CC>
struct LnLanes {
  static constexpr int LPR = CC / 8, RPW = 32 / LPR;
  static_assert(CC == 64 || CC == 128 || CC == 256, "channels");
};

__device__ __forceinline__ void unpack8(const uint4 &w, float (&v)[8]) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) v[2 * j] = lo_bf(ww[j]), v[2 * j + 1] = hi_bf(ww[j]);
}

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// The HM per-lane values v[h] summed over a lane group of LPR lanes (LPR >= HM), by recursive
// halving: at each of the first log2(HM) levels a lane keeps half of its heads and receives the
// partner's partial sums of them, then plain xor steps finish. Returns the sum for head
// head_of_lane<LPR, HM>(sl); a fixed tree, HM - 1 + log2(LPR / HM) shuffles instead of HM log2(LPR).
template <int LPR, int HM>
__device__ __forceinline__ float group_sum_scatter(float (&v)[HM], int sl) {
  int count = HM;
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) {
    if (count > 1) {
      const int half = count / 2;
      const bool upper = (sl & o) != 0;
#pragma unroll
      for (int i = 0; i < HM / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half], keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      count = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

// The head whose sum group_sum_scatter leaves in lane sl of its group.
template <int LPR, int HM>
__device__ __forceinline__ int head_of_lane(int sl) {
  int h = 0, w = HM / 2;
#pragma unroll
  for (int o = LPR / 2; o > 0 && w > 0; o >>= 1, w >>= 1)
    if (sl & o) h += w;
  return h;
}

template <int CC, int HM>
__global__ void __launch_bounds__(256) mod_ln_fwd_kernel(const uint16_t *__restrict__ z, const float *__restrict__ gamma,
                                                         const float *__restrict__ beta, const uint16_t *__restrict__ wb,
                                                         int H, int N, int node, float eps, int64_t M,
                                                         uint16_t *__restrict__ zt, float *__restrict__ mu,
                                                         float *__restrict__ rstd, uint16_t *__restrict__ bias) {
  using L = LnLanes<CC>;
  const int lane = threadIdx.x & 31, sl = lane % L::LPR, rs = lane / L::LPR;
  const int64_t w0 = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5), ws = (int64_t)gridDim.x * 8;
  float gm[8], bt[8], wv[HM][8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    gm[j] = gamma[sl * 8 + j];
    bt[j] = beta[sl * 8 + j];
  }
#pragma unroll
  for (int h = 0; h < HM; ++h) {
    if (h < H) {
      unpack8(*reinterpret_cast<const uint4 *>(wb + h * CC + sl * 8), wv[h]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) wv[h][j] = 0.f;
    }
  }
  const int64_t NN = (int64_t)N * N;
  const uint32_t nn32 = (uint32_t)NN, n32 = (uint32_t)N;
  // U position groups per warp at a time, their loads issued together (bytes in flight)
  constexpr int U = 4;
  for (int64_t g = w0 * U; g * L::RPW < M; g += ws * U) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t m = (g + u) * L::RPW + rs;
      raw[u] = m < M ? *reinterpret_cast<const uint4 *>(z + m * CC + sl * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
    // (b, x, y) of the first group's position by division, the others by stepping (positions and
    // N^2 fit 32 bits: B N <= 65535, N <= 1024)
    uint32_t pb, px, py;
    {
      const uint32_t m32 = (uint32_t)(g * L::RPW + rs);
      pb = m32 / nn32;
      px = (m32 - pb * nn32) / n32;
      py = m32 - pb * nn32 - px * n32;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t m = (g + u) * L::RPW + rs;
      const bool live = m < M;  // (lane groups past the last position idle, but join the shuffles)
      if (u > 0) {
        py += L::RPW;  // (RPW <= 4 < N: at most one carry)
        if (py >= n32) {
          py -= n32;
          if (++px == n32) {
            px = 0;
            ++pb;
          }
        }
      }
      float x[8];
      unpack8(raw[u], x);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) s += x[j];
      const float mean = group_sum<L::LPR>(s) * (1.f / CC);
      float q = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) q = fmaf(x[j] - mean, x[j] - mean, q);
      const float r = rsqrtf(group_sum<L::LPR>(q) * (1.f / CC) + eps);
      uint32_t yw[4];
      float y[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        yw[j] = pack_bf16x2(fmaf((x[2 * j] - mean) * r, gm[2 * j], bt[2 * j]),
                            fmaf((x[2 * j + 1] - mean) * r, gm[2 * j + 1], bt[2 * j + 1]));
        y[2 * j] = lo_bf(yw[j]);
        y[2 * j + 1] = hi_bf(yw[j]);
      }
      if (live) {
        *reinterpret_cast<uint4 *>(zt + m * CC + sl * 8) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
        if (sl == 0) {
          mu[m] = mean;
          rstd[m] = r;
        }
      }
      const int64_t boff = node == 0 ? (int64_t)px * N + py : (int64_t)py * N + px;
      float p[HM];
#pragma unroll
      for (int h = 0; h < HM; ++h) {
        p[h] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) p[h] = fmaf(y[j], wv[h][j], p[h]);
      }
      const float ph = group_sum_scatter<L::LPR, HM>(p, sl);
      const int hh = head_of_lane<L::LPR, HM>(sl);
      if (live && hh < H && (sl & (L::LPR / HM - 1)) == 0)
        bias[((int64_t)pb * H + hh) * NN + boff] = (uint16_t)(pack_bf16x2(ph, 0.f) & 0xffffu);
    }
  }
}

// ================================================================ gate: go = sigmoid(gl) O
__global__ void __launch_bounds__(256) mod_gate_kernel(const uint16_t *__restrict__ gl, const uint16_t *__restrict__ O,
                                                       uint16_t *__restrict__ go, int64_t chunks) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < chunks; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 g = reinterpret_cast<const uint4 *>(gl)[i], o = reinterpret_cast<const uint4 *>(O)[i];
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, ow[4] = {o.x, o.y, o.z, o.w};
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      r[j] = pack_bf16x2(sigm(lo_bf(gw[j])) * lo_bf(ow[j]), sigm(hi_bf(gw[j])) * hi_bf(ow[j]));
    reinterpret_cast<uint4 *>(go)[i] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// ================================================================ LayerNorm backward
// One CTA per fixed chunk of `rpc` pair positions; lane groups as in the forward (CC / 8 lanes per
// position, 8 channels per lane), the warps of the CTA taking the chunk's positions in turn, U
// positions per lane group at a time with their loads issued together. g = dzt + sum_h dbias_h wb[h]
// is the full gradient of zt; with zh = (z - mean) rstd and dzh = g gamma,
// dz = rstd (dzh - mean(dzh) - zh mean(dzh zh)). The CTA's partial sums of dgamma (g zh), dbeta (g)
// and dwb[h] (dbias_h zt) are added over the lane groups of a warp by a fixed xor-shuffle tree, then
// over the warps in warp order, and written to part[blockIdx.x][2 + H][CC]. gamma and wb are read
// from shared memory (broadcast loads), which keeps the kernel at two CTAs per SM for H <= 4.
template <int CC, int HM>
__global__ void __launch_bounds__(256, HM <= 4 ? 2 : 1) mod_ln_bwd_kernel(const float *__restrict__ dzt, const uint16_t *__restrict__ dbias,
                                                            const uint16_t *__restrict__ z, const uint16_t *__restrict__ zt,
                                                            const float *__restrict__ mu, const float *__restrict__ rstd,
                                                            const float *__restrict__ gamma, const uint16_t *__restrict__ wb,
                                                            int H, int N, int node, int64_t M, int rpc,
                                                            uint16_t *__restrict__ dz, float *__restrict__ part) {
  using L = LnLanes<CC>;
  constexpr int U = 1;  // (more positions in flight per lane group cost the second CTA per SM)
  __shared__ __align__(16) float red[(2 + HM) * CC];
  __shared__ __align__(16) float sw[(1 + HM) * CC];  // gamma, then wb[h] in FP32
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, sl = lane % L::LPR, rs = lane / L::LPR;
  const int gbase = lane - sl;  // first lane of this lane group
  for (int i = threadIdx.x; i < (1 + HM) * CC; i += blockDim.x) {
    const int h = i / CC - 1, cc = i % CC;
    sw[i] = h < 0 ? gamma[cc] : (h < H ? __uint_as_float((uint32_t)wb[h * CC + cc] << 16) : 0.f);
  }
  __syncthreads();
  float ag[8], ab[8], aw[HM][8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ag[j] = 0.f;
    ab[j] = 0.f;
#pragma unroll
    for (int h = 0; h < HM; ++h) aw[h][j] = 0.f;
  }
  const int64_t NN = (int64_t)N * N;
  const int64_t r0 = (int64_t)blockIdx.x * rpc, r1 = min(M, r0 + rpc);
  const int step = 8 * U * L::RPW;  // positions a lane group advances per iteration
  // (b, x, y) of this lane group's U positions, advanced incrementally (positions fit 32 bits)
  uint32_t pb[U], px[U], py[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint32_t m = (uint32_t)(r0 + (int64_t)warp * U * L::RPW + u * L::RPW + rs), nn = (uint32_t)NN;
    pb[u] = m / nn;
    px[u] = (m - pb[u] * nn) / (uint32_t)N;
    py[u] = m - pb[u] * nn - px[u] * (uint32_t)N;
  }
  for (int64_t g0 = r0 + (int64_t)warp * U * L::RPW; g0 < r1; g0 += step) {
    float4 rg[U][2];
    uint4 rz[U], rt[U];
    float rdb[U], rmu[U], rr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t m = g0 + u * L::RPW + rs;
      if (m < r1) {
        const int64_t boff = node == 0 ? (int64_t)px[u] * N + py[u] : (int64_t)py[u] * N + px[u];
        // lane h of the group loads dbias of head h
        rdb[u] = sl < H ? __uint_as_float((uint32_t)dbias[((int64_t)pb[u] * H + sl) * NN + boff] << 16) : 0.f;
        rg[u][0] = *reinterpret_cast<const float4 *>(dzt + m * CC + sl * 8);
        rg[u][1] = *reinterpret_cast<const float4 *>(dzt + m * CC + sl * 8 + 4);
        rz[u] = *reinterpret_cast<const uint4 *>(z + m * CC + sl * 8);
        rt[u] = *reinterpret_cast<const uint4 *>(zt + m * CC + sl * 8);
        rmu[u] = mu[m];
        rr[u] = rstd[m];
      } else {  // past the chunk: zeros, which add nothing (the group still joins the shuffles)
        rdb[u] = 0.f;
        rg[u][0] = rg[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        rz[u] = rt[u] = make_uint4(0u, 0u, 0u, 0u);
        rmu[u] = 0.f;
        rr[u] = 0.f;
      }
      py[u] += step;
      while (py[u] >= (uint32_t)N) {
        py[u] -= N;
        if (++px[u] == (uint32_t)N) {
          px[u] = 0;
          ++pb[u];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t m = g0 + u * L::RPW + rs;
      float db[HM];
#pragma unroll
      for (int h = 0; h < HM; ++h) db[h] = __shfl_sync(0xffffffffu, rdb[u], gbase + (h < H ? h : 0));
      float g[8], zv[8], tv[8];
      g[0] = rg[u][0].x, g[1] = rg[u][0].y, g[2] = rg[u][0].z, g[3] = rg[u][0].w;
      g[4] = rg[u][1].x, g[5] = rg[u][1].y, g[6] = rg[u][1].z, g[7] = rg[u][1].w;
      unpack8(rz[u], zv);
      unpack8(rt[u], tv);
#pragma unroll
      for (int h = 0; h < HM; ++h) {
        if (h >= H) break;
        const float4 w0 = *reinterpret_cast<const float4 *>(sw + (1 + h) * CC + sl * 8);
        const float4 w1 = *reinterpret_cast<const float4 *>(sw + (1 + h) * CC + sl * 8 + 4);
        g[0] = fmaf(db[h], w0.x, g[0]), g[1] = fmaf(db[h], w0.y, g[1]), g[2] = fmaf(db[h], w0.z, g[2]);
        g[3] = fmaf(db[h], w0.w, g[3]), g[4] = fmaf(db[h], w1.x, g[4]), g[5] = fmaf(db[h], w1.y, g[5]);
        g[6] = fmaf(db[h], w1.z, g[6]), g[7] = fmaf(db[h], w1.w, g[7]);
      }
      const float4 g0v = *reinterpret_cast<const float4 *>(sw + sl * 8);
      const float4 g1v = *reinterpret_cast<const float4 *>(sw + sl * 8 + 4);
      const float gm[8] = {g0v.x, g0v.y, g0v.z, g0v.w, g1v.x, g1v.y, g1v.z, g1v.w};
      const float mean = rmu[u], r = rr[u];
      float zh[8], dzh[8], s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        zh[j] = (zv[j] - mean) * r;
        dzh[j] = g[j] * gm[j];
        s1 += dzh[j];
        s2 = fmaf(dzh[j], zh[j], s2);
      }
      s1 = group_sum<L::LPR>(s1) * (1.f / CC);
      s2 = group_sum<L::LPR>(s2) * (1.f / CC);
      if (m < r1) {
        uint32_t ow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ow[j] = pack_bf16x2(r * (dzh[2 * j] - s1 - zh[2 * j] * s2), r * (dzh[2 * j + 1] - s1 - zh[2 * j + 1] * s2));
        *reinterpret_cast<uint4 *>(dz + m * CC + sl * 8) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      // (positions past the chunk carry zeros: they add nothing)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ag[j] = fmaf(g[j], zh[j], ag[j]);
        ab[j] += g[j];
#pragma unroll
        for (int h = 0; h < HM; ++h) aw[h][j] = fmaf(db[h], tv[j], aw[h][j]);
      }
    }
  }
  // the warp's lane groups added by a fixed xor tree (every lane group ends with the warp's sums)
#pragma unroll
  for (int o = L::LPR; o < 32; o <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ag[j] += __shfl_xor_sync(0xffffffffu, ag[j], o);
      ab[j] += __shfl_xor_sync(0xffffffffu, ab[j], o);
#pragma unroll
      for (int h = 0; h < HM; ++h) aw[h][j] += __shfl_xor_sync(0xffffffffu, aw[h][j], o);
    }
  }
  // then the warps in warp order
  const int nrow = 2 + H;
  for (int w = 0; w < 8; ++w) {
    if (warp == w && rs == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = sl * 8 + j;
        red[c] = w ? red[c] + ag[j] : ag[j];
        red[CC + c] = w ? red[CC + c] + ab[j] : ab[j];
#pragma unroll
        for (int h = 0; h < HM; ++h)
          if (h < H) red[(2 + h) * CC + c] = w ? red[(2 + h) * CC + c] + aw[h][j] : aw[h][j];
      }
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < nrow * CC; i += blockDim.x) part[(int64_t)blockIdx.x * nrow * CC + i] = red[i];
}

// ================================================================ ordered sum of partials
// out[i] = sum over t of part[t][i], for i < n, in a fixed order: a CTA takes 32 consecutive i
// (threadIdx.x) and 8 lanes of t (threadIdx.y); lane y adds t = y, y + 8, y + 16, ... in increasing
// t, then the 8 lane sums are added in lane order. The result is written in up to three pieces:
// i < n0 to o0, i < n0 + n1 to o1, the rest to o2.
__global__ void __launch_bounds__(256) mod_reduce_kernel(const float *__restrict__ part, int T, int64_t n, float *o0,
                                                         int64_t n0, float *o1, int64_t n1, float *o2) {
  __shared__ float acc[8][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int64_t i = (int64_t)blockIdx.x * 32 + tx;
  float s = 0.f;
  if (i < n) {
    int t = ty;
    for (; t + 24 < T; t += 32) {  // four loads in flight, added in t order
      const float a0 = part[(int64_t)t * n + i], a1 = part[(int64_t)(t + 8) * n + i];
      const float a2 = part[(int64_t)(t + 16) * n + i], a3 = part[(int64_t)(t + 24) * n + i];
      s = (((s + a0) + a1) + a2) + a3;
    }
    for (; t < T; t += 8) s += part[(int64_t)t * n + i];
  }
  acc[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && i < n) {
    float r = acc[0][tx];
#pragma unroll
    for (int y = 1; y < 8; ++y) r += acc[y][tx];
    if (i < n0)
      o0[i] = r;
    else if (i < n0 + n1)
      o1[i - n0] = r;
    else
      o2[i - n0 - n1] = r;
  }
}

// ================================================================ host side
constexpr size_t kAlign = 256;
size_t aup(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const tri_module_shape &s) {
  if (s.B < 1 || s.N < 1 || s.c < 1 || s.H < 1 || s.d < 1 || !(s.eps > 0.f) || !isfinite(s.eps) ||
      (s.node != TRI_ATTN_NODE_STARTING && s.node != TRI_ATTN_NODE_ENDING))
    return TRI_ATTN_ERR_INVALID_ARG;
  if ((s.c != 64 && s.c != 128 && s.c != 256) || (s.d != 16 && s.d != 32) || s.H > 8 || (s.H * s.d) % 64 ||
      s.N < 16 || s.N > TRI_ATTN_MAX_N || (int64_t)s.B * s.N > 65535)
    return TRI_ATTN_ERR_UNSUPPORTED;
  return TRI_ATTN_OK;
}

tri_attn_shape attn_shape(const tri_module_shape &s) {
  return tri_attn_shape{s.B, s.N, s.N, s.H, s.d, 1.f / sqrtf((float)s.d), s.node};
}

int64_t rows_of(const tri_module_shape &s) { return (int64_t)s.B * s.N * s.N; }

// Fixed chunks of pair positions for the sums over positions: about 144 chunks of a multiple of
// 64 rows (the GEMM's K step), chosen from the shape alone.
int split_rows(int64_t M) { return (int)std::max<int64_t>(64, ((M + 143) / 144 + 63) / 64 * 64); }
int ln_rows(int64_t M) { return (int)std::max<int64_t>(8, ((M + 303) / 304 + 7) / 8 * 8); }

struct SavedLayout {
  size_t zt, mu, rstd, q, k, v, gl, bias, O, Ores, LSE, go, total;
};

SavedLayout saved_layout(const tri_module_shape &s) {
  const size_t M = (size_t)rows_of(s), hd = (size_t)s.H * s.d;
  const size_t act = aup(2 * M * hd);
  SavedLayout L;
  L.zt = 0;
  L.mu = aup(2 * M * s.c);
  L.rstd = L.mu + aup(4 * M);
  L.q = L.rstd + aup(4 * M);
  L.k = L.q + act;
  L.v = L.k + act;
  L.gl = L.v + act;
  L.bias = L.gl + act;
  L.O = L.bias + aup(2 * (size_t)s.B * s.H * s.N * s.N);
  L.Ores = L.O + act;
  L.LSE = L.Ores + act;
  L.go = L.LSE + aup(4 * (size_t)s.B * s.N * s.H * s.N);
  L.total = L.go + act;
  return L;
}

struct BwdLayout {
  size_t dO, dgl, dq, dk, dv, dbias, dzt, attn, pWo, pW, pLN, total;
  size_t attn_bytes;
  int Kc, Tsplit, rpc, nln;
};

BwdLayout bwd_layout(const tri_module_shape &s) {
  const size_t M = (size_t)rows_of(s), hd = (size_t)s.H * s.d;
  const size_t act = aup(2 * M * hd);
  BwdLayout L;
  L.Kc = split_rows((int64_t)M);
  L.Tsplit = (int)((M + L.Kc - 1) / L.Kc);
  L.rpc = ln_rows((int64_t)M);
  L.nln = (int)((M + L.rpc - 1) / L.rpc);
  L.attn_bytes = tri_attn_bwd_workspace_size(attn_shape(s));
  L.dO = 0;
  L.dgl = act;
  L.dq = 2 * act;
  L.dk = 3 * act;
  L.dv = 4 * act;
  L.dbias = 5 * act;
  L.dzt = L.dbias + aup(2 * (size_t)s.B * s.H * s.N * s.N);
  L.attn = L.dzt + aup(4 * M * s.c);
  L.pWo = L.attn + aup(L.attn_bytes);
  L.pW = L.pWo + aup(4 * (size_t)L.Tsplit * s.c * hd);
  L.pLN = L.pW + aup(4 * (size_t)L.Tsplit * 4 * hd * s.c);
  L.total = L.pLN + aup(4 * (size_t)L.nln * (2 + s.H) * s.c);
  return L;
}

template <typename T>
T *at(void *base, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(base) + off);
}

template <int HM>
void ln_fwd_c(const tri_module_shape &s, int grid, const uint16_t *z, const float *gamma, const float *beta,
              const uint16_t *wb, uint16_t *zt, float *mu, float *rstd, uint16_t *bias, cudaStream_t st) {
  const int64_t M = rows_of(s);
  switch (s.c) {
    case 64: mod_ln_fwd_kernel<64, HM><<<grid, 256, 0, st>>>(z, gamma, beta, wb, s.H, s.N, s.node, s.eps, M, zt, mu, rstd, bias); break;
    case 128: mod_ln_fwd_kernel<128, HM><<<grid, 256, 0, st>>>(z, gamma, beta, wb, s.H, s.N, s.node, s.eps, M, zt, mu, rstd, bias); break;
    default: mod_ln_fwd_kernel<256, HM><<<grid, 256, 0, st>>>(z, gamma, beta, wb, s.H, s.N, s.node, s.eps, M, zt, mu, rstd, bias); break;
  }
}

cudaError_t launch_ln_fwd(const tri_module_shape &s, const uint16_t *z, const float *gamma, const float *beta,
                          const uint16_t *wb, uint16_t *zt, float *mu, float *rstd, uint16_t *bias, cudaStream_t st) {
  const int64_t M = rows_of(s);
  const int rpw = 32 / (s.c / 8);  // positions per warp at a time
  const int grid = (int)std::min<int64_t>((M + 32 * rpw - 1) / (32 * rpw), 152 * 16);
  if (s.H <= 4)
    ln_fwd_c<4>(s, grid, z, gamma, beta, wb, zt, mu, rstd, bias, st);
  else
    ln_fwd_c<8>(s, grid, z, gamma, beta, wb, zt, mu, rstd, bias, st);
  return cudaGetLastError();
}

template <int HM>
void ln_bwd_c(const tri_module_shape &s, const BwdLayout &L, const float *dzt, const uint16_t *dbias, const uint16_t *z,
              const uint16_t *zt, const float *mu, const float *rstd, const float *gamma, const uint16_t *wb,
              uint16_t *dz, float *part, cudaStream_t st) {
  const int64_t M = rows_of(s);
  switch (s.c) {
    case 64: mod_ln_bwd_kernel<64, HM><<<L.nln, 256, 0, st>>>(dzt, dbias, z, zt, mu, rstd, gamma, wb, s.H, s.N, s.node, M, L.rpc, dz, part); break;
    case 128: mod_ln_bwd_kernel<128, HM><<<L.nln, 256, 0, st>>>(dzt, dbias, z, zt, mu, rstd, gamma, wb, s.H, s.N, s.node, M, L.rpc, dz, part); break;
    default: mod_ln_bwd_kernel<256, HM><<<L.nln, 256, 0, st>>>(dzt, dbias, z, zt, mu, rstd, gamma, wb, s.H, s.N, s.node, M, L.rpc, dz, part); break;
  }
}

cudaError_t launch_ln_bwd(const tri_module_shape &s, const BwdLayout &L, const float *dzt, const uint16_t *dbias,
                          const uint16_t *z, const uint16_t *zt, const float *mu, const float *rstd, const float *gamma,
                          const uint16_t *wb, uint16_t *dz, float *part, cudaStream_t st) {
  if (s.H <= 4)
    ln_bwd_c<4>(s, L, dzt, dbias, z, zt, mu, rstd, gamma, wb, dz, part, st);
  else
    ln_bwd_c<8>(s, L, dzt, dbias, z, zt, mu, rstd, gamma, wb, dz, part, st);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const float *part, int T, int64_t n, float *o0, int64_t n0, float *o1, int64_t n1, float *o2,
                          cudaStream_t st) {
  mod_reduce_kernel<<<(unsigned)((n + 31) / 32), dim3(32, 8), 0, st>>>(part, T, n, o0, n0, o1 ? o1 : o0, n1,
                                                                      o2 ? o2 : o0);
  return cudaGetLastError();
}

cudaError_t mark_ok(cudaError_t e, int k, cudaStream_t st) { return e == cudaSuccess ? timing_mark(k, st) : e; }

}  // namespace
}  // namespace triattn

using namespace triattn;

extern "C" {

size_t tri_module_saved_size(tri_module_shape shape) {
  if (check_shape(shape)) return 0;
  return saved_layout(shape).total;
}

size_t tri_module_bwd_workspace_size(tri_module_shape shape) {
  if (check_shape(shape)) return 0;
  const BwdLayout L = bwd_layout(shape);
  return L.attn_bytes ? L.total : 0;
}

int tri_module_fwd(tri_module_shape shape, const tri_attn_bf16 *z, const float *gamma, const float *beta,
                   const tri_attn_bf16 *W, const tri_attn_bf16 *wb, const tri_attn_bf16 *Wo,
                   const tri_attn_bf16 *mask, tri_attn_bf16 *out, void *saved, size_t saved_bytes, void *stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  const void *ptrs[] = {z, gamma, beta, W, wb, Wo, out, saved};
  for (const void *p : ptrs) {
    if (!p) return TRI_ATTN_ERR_INVALID_ARG;
    if (!aligned16(p)) return TRI_ATTN_ERR_UNSUPPORTED;
  }
  if (mask && !aligned16(mask)) return TRI_ATTN_ERR_UNSUPPORTED;
  const SavedLayout L = saved_layout(shape);
  if (saved_bytes < L.total) return TRI_ATTN_ERR_WORKSPACE;
  const int64_t M = rows_of(shape);
  const int hd = shape.H * shape.d, c = shape.c;
  uint16_t *zt = at<uint16_t>(saved, L.zt), *q = at<uint16_t>(saved, L.q), *k = at<uint16_t>(saved, L.k),
           *v = at<uint16_t>(saved, L.v), *gl = at<uint16_t>(saved, L.gl), *bias = at<uint16_t>(saved, L.bias),
           *O = at<uint16_t>(saved, L.O), *Ores = at<uint16_t>(saved, L.Ores), *go = at<uint16_t>(saved, L.go);
  float *mu = at<float>(saved, L.mu), *rstd = at<float>(saved, L.rstd), *LSE = at<float>(saved, L.LSE);
  int *status = device_status_word();
  if (!status) return TRI_ATTN_ERR_CUDA;
  // every plan before the first launch
  MGemm<false, false, kOutBF16> g_in, g_out;
  const uint16_t *a_in[1] = {zt}, *a_out[1] = {go};
  if (g_in.plan(a_in, 1, c, W, (int)M, 4 * hd, c, c, out_bf16(q, k, v, gl, hd)) != cudaSuccess ||
      g_out.plan(a_out, 1, hd, Wo, (int)M, c, hd, hd, out_bf16(out, nullptr, nullptr, nullptr, c)) != cudaSuccess)
    return TRI_ATTN_ERR_CUDA;
  AttnFwdCall ac;
  rc = attn_fwd_prepare(attn_shape(shape), q, k, v, bias, mask, O, LSE, Ores, &ac);
  if (rc) return rc;
  auto st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_ln_fwd(shape, z, gamma, beta, wb, zt, mu, rstd, bias, st);
  e = mark_ok(e, 0, st);
  if (e == cudaSuccess) e = g_in.launch(status, st);
  e = mark_ok(e, 1, st);
  if (e == cudaSuccess) e = attn_fwd_enqueue(ac, 2, st);
  if (e == cudaSuccess) {
    const int64_t chunks = M * hd / 8;
    mod_gate_kernel<<<(int)std::min<int64_t>((chunks + 255) / 256, 152 * 8), 256, 0, st>>>(gl, O, go, chunks);
    e = cudaGetLastError();
  }
  e = mark_ok(e, 4, st);
  if (e == cudaSuccess) e = g_out.launch(status, st);
  e = mark_ok(e, 5, st);
  return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA;
}

int tri_module_bwd(tri_module_shape shape, const tri_attn_bf16 *z, const float *gamma, const float *beta,
                   const tri_attn_bf16 *W, const tri_attn_bf16 *wb, const tri_attn_bf16 *Wo,
                   const tri_attn_bf16 *mask, const void *saved, size_t saved_bytes, const tri_attn_bf16 *dout,
                   tri_attn_bf16 *dz, float *dgamma, float *dbeta, float *dW, float *dwb, float *dWo,
                   void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  const void *ptrs[] = {z, gamma, beta, W, wb, Wo, saved, dout, dz, dgamma, dbeta, dW, dwb, dWo, workspace};
  for (const void *p : ptrs) {
    if (!p) return p == workspace ? TRI_ATTN_ERR_WORKSPACE : TRI_ATTN_ERR_INVALID_ARG;
    if (!aligned16(p)) return TRI_ATTN_ERR_UNSUPPORTED;
  }
  if (mask && !aligned16(mask)) return TRI_ATTN_ERR_UNSUPPORTED;
  const SavedLayout S = saved_layout(shape);
  if (saved_bytes < S.total) return TRI_ATTN_ERR_WORKSPACE;
  const BwdLayout L = bwd_layout(shape);
  if (!L.attn_bytes) return TRI_ATTN_ERR_CUDA;
  if (workspace_bytes < L.total) return TRI_ATTN_ERR_WORKSPACE;
  const int64_t M = rows_of(shape);
  const int hd = shape.H * shape.d, c = shape.c, H = shape.H;
  void *sv = const_cast<void *>(saved);
  const uint16_t *zt = at<uint16_t>(sv, S.zt), *q = at<uint16_t>(sv, S.q), *k = at<uint16_t>(sv, S.k),
                 *v = at<uint16_t>(sv, S.v), *gl = at<uint16_t>(sv, S.gl), *bias = at<uint16_t>(sv, S.bias),
                 *O = at<uint16_t>(sv, S.O), *Ores = at<uint16_t>(sv, S.Ores), *go = at<uint16_t>(sv, S.go);
  const float *mu = at<float>(sv, S.mu), *rstd = at<float>(sv, S.rstd), *LSE = at<float>(sv, S.LSE);
  uint16_t *dO = at<uint16_t>(workspace, L.dO), *dgl = at<uint16_t>(workspace, L.dgl),
           *dq = at<uint16_t>(workspace, L.dq), *dk = at<uint16_t>(workspace, L.dk), *dv = at<uint16_t>(workspace, L.dv),
           *dbias = at<uint16_t>(workspace, L.dbias);
  float *dzt = at<float>(workspace, L.dzt), *pWo = at<float>(workspace, L.pWo), *pW = at<float>(workspace, L.pW),
        *pLN = at<float>(workspace, L.pLN);
  int *status = device_status_word();
  if (!status) return TRI_ATTN_ERR_CUDA;
  // every plan before the first launch
  MGemm<false, true, kOutGate> g_dgo;   // dgo[m][j] = sum_c dout[m][c] Wo[c][j]
  MGemm<true, true, kOutF32> g_dwo;     // dWo[c][j] = sum_m dout[m][c] go[m][j]
  MGemm<false, true, kOutF32> g_dzt;    // dzt[m][c] = sum_r dproj[m][r] W[r][c]
  MGemm<true, true, kOutF32> g_dw;      // dW[r][c] = sum_m dproj[m][r] zt[m][c]
  const uint16_t *a_dout[1] = {dout}, *a_proj[4] = {dq, dk, dv, dgl};
  MGemmArgs gate{}, f_wo{}, f_zt{}, f_w{};
  gate.P = O;
  gate.G = gl;
  gate.dP = dO;
  gate.dG = dgl;
  f_wo.D0 = pWo;
  f_zt.D0 = dzt;
  f_w.D0 = pW;
  if (g_dgo.plan(a_dout, 1, c, Wo, (int)M, hd, c, c, gate) != cudaSuccess ||
      g_dwo.plan(a_dout, 1, c, go, c, hd, (int)M, L.Kc, f_wo) != cudaSuccess ||
      g_dzt.plan(a_proj, 4, hd, W, (int)M, c, 4 * hd, 4 * hd, f_zt) != cudaSuccess ||
      g_dw.plan(a_proj, 4, hd, zt, 4 * hd, c, (int)M, L.Kc, f_w) != cudaSuccess)
    return TRI_ATTN_ERR_CUDA;
  AttnBwdCall ac;
  rc = attn_bwd_prepare(attn_shape(shape), q, k, v, bias, mask, O, Ores, LSE, dO, dq, dk, dv, dbias,
                        at<void>(workspace, L.attn), L.attn_bytes, &ac);
  if (rc) return rc;
  auto st = static_cast<cudaStream_t>(stream);
  cudaError_t e = g_dgo.launch(status, st);
  e = mark_ok(e, 0, st);
  if (e == cudaSuccess) e = g_dwo.launch(status, st);
  e = mark_ok(e, 1, st);
  if (e == cudaSuccess) e = launch_reduce(pWo, L.Tsplit, (int64_t)c * hd, dWo, (int64_t)c * hd, nullptr, 0, nullptr, st);
  e = mark_ok(e, 2, st);
  if (e == cudaSuccess) e = attn_bwd_enqueue(ac, 3, st);
  if (e == cudaSuccess) e = g_dzt.launch(status, st);
  e = mark_ok(e, 7, st);
  if (e == cudaSuccess) e = launch_ln_bwd(shape, L, dzt, dbias, z, zt, mu, rstd, gamma, wb, dz, pLN, st);
  e = mark_ok(e, 8, st);
  if (e == cudaSuccess) e = launch_reduce(pLN, L.nln, (int64_t)(2 + H) * c, dgamma, c, dbeta, c, dwb, st);
  e = mark_ok(e, 9, st);
  if (e == cudaSuccess) e = g_dw.launch(status, st);
  e = mark_ok(e, 10, st);
  if (e == cudaSuccess)
    e = launch_reduce(pW, L.Tsplit, (int64_t)4 * hd * c, dW, (int64_t)4 * hd * c, nullptr, 0, nullptr, st);
  e = mark_ok(e, 11, st);
  return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA;
}

}  // extern "C"
