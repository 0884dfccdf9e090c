// Triangle multiplicative update: element-wise gating, the triangular contraction and its
// gradients (the fast_trimul article on kongchang.com, section "什么是三角乘法更新": gating, an
// outer product of two gated operands and a reduction along one axis of the pair
// representation; TurboPairFormer, arXiv 2610.05854v1, Abstract: the triangle multiplication
// kernels used beside the attention).
//
//   a = sigmoid(G_a) P_a,  b = sigmoid(G_b) P_b      (stored in BF16)
//   outgoing:  X[b,i,j,c] = sum_k a[b,i,k,c] b[b,j,k,c]
//   incoming:  X[b,i,j,c] = sum_k a[b,k,i,c] b[b,k,j,c]
//
// The contraction is one N x N matrix product per (batch, channel), so the gated operands are
// stored channel-major, [B, C, N, N]. Two layouts of the projections and their gradients:
//
// - pair layout [B, N, N, C] (channels innermost): the gating kernel transposes while it gates,
//   A[b,c,i,k] = a[b,i,k,c] for the outgoing update and a[b,k,i,c] for the incoming one (the pair
//   axes swapped), likewise B, so both directions are X_bc = A_bc B_bc^T with K-major operands.
//   The backward products dA_bc = dX_bc B_bc and dB_bc = dX_bc^T A_bc are the same GEMM with one
//   or both operands read MN-major (the tensor cores' transposed operand mode, no transposed
//   copies), written in FP32 to a workspace, and a gradient kernel maps them back to the pair
//   layout while applying the gating gradient.
// - channel-major layout [B, C, N, N]: gating is element-wise; the incoming update reads its
//   operands MN-major instead (X_bc = A_bc^T B_bc), and each backward product applies the gating
//   gradient in its epilogue, so dA and dB never reach memory.
//
// Gating is bound by HBM bandwidth (one read of P and G, one write of the operand); folding it
// into the GEMM's operand loads would recompute each sigmoid once per output tile that reads it
// (N / 256 or N / 128 times), which costs more on the MUFU pipe than the extra HBM pass.
#include <algorithm>

#include "common.cuh"
#include "launch.cuh"
#include "sm100.cuh"
#include "sync.cuh"
#include "tmap.cuh"
#include "tri_mul.h"

namespace triattn {
using namespace sm100;

cudaError_t timing_mark(int k, cudaStream_t st);
int *device_status_word();

namespace {

// sigmoid in FP32 from the fast exponential and reciprocal: relative error a few FP32 ulp plus
// about one per unit of |x| (the fast exponential's error grows with its argument); 0 below
// x = -87, where 1 + exp(-x) leaves the reciprocal's range.
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

constexpr int kGateT = 16, kGateThreads = 256;  // positions per tile side, threads per CTA

// Both pair-layout gating kernels run a 1-D grid of (batch, r tile, s tile, channel group,
// operand) with the operand and then the channel group varying fastest: the CTAs that read the
// same pair positions (their channel groups share cache lines) run at the same time.
__device__ __forceinline__ void tile_of(int N, int groups, int &op, int &grp, int &b, int &r0, int &s0) {
  const int nt = (N + kGateT - 1) / kGateT;
  int u = blockIdx.x;
  op = u & 1;
  u >>= 1;
  grp = u % groups;
  u /= groups;
  s0 = (u % nt) * kGateT;
  u /= nt;
  r0 = (u % nt) * kGateT;
  b = u / nt;
}

// ---------------------------------------------------------------- gating: pair -> channel-major
// One CTA: 16 x 16 output positions (r, s) and a group of up to 64 channels, for one of the two
// operands. Input position (x, y) = (r, s), or (s, r) when the operand is transposed (incoming
// update). Each thread reads 16 channel bytes
// of two neighbouring positions s, s + 1 and writes the gated pairs as 32-bit words
// (a(s), a(s + 1)) into shared memory [channel][r][s / 2]; the channel stride (145 words) and
// row pitch (9 words) keep both the scattered writes and the row reads free of most bank
// conflicts. Output rows (c, r) of 16 values (32 bytes) are then stored with 16-byte stores.
constexpr int kGateCG = 64;                    // channels per CTA
constexpr int kGateRowW = 9, kGateChW = 145;  // words
constexpr int kGateSmem = kGateCG * kGateChW * 4;

struct GateArgs {
  const uint16_t *P[2], *G[2];
  uint16_t *out[2];
  int N, C, groups, transposed;
};

__global__ void __launch_bounds__(kGateThreads) trimul_gate_kernel(const GateArgs g) {
  extern __shared__ uint32_t tw[];  // [64][145] words
  int op, grp, b, r0, s0;
  tile_of(g.N, g.groups, op, grp, b, r0, s0);
  const int N = g.N, C = g.C, c0 = grp * kGateCG, nq = min(kGateCG, C - c0) / 8;
  const uint4 *P = reinterpret_cast<const uint4 *>(op ? g.P[1] : g.P[0]),
              *G = reinterpret_cast<const uint4 *>(op ? g.G[1] : g.G[0]);
  const int64_t cv = C / 8;
#pragma unroll 2
  for (int e = threadIdx.x; e < kGateT * 8 * 8; e += kGateThreads) {
    const int q = e & 7, sp = (e >> 3) & 7, rl = e >> 6;
    if (q >= nq) continue;
    const int r = r0 + rl, s = s0 + 2 * sp;
    uint4 p0 = make_uint4(0, 0, 0, 0), g0 = p0, p1 = p0, g1 = p0;
    if (r < N && s < N) {  // N is even: s + 1 < N as well
      const int64_t i0 = g.transposed ? ((int64_t)b * N + s) * N + r : ((int64_t)b * N + r) * N + s;
      const int64_t i1 = g.transposed ? i0 + N : i0 + 1;
      const int64_t o = c0 / 8 + q;
      p0 = P[i0 * cv + o], g0 = G[i0 * cv + o], p1 = P[i1 * cv + o], g1 = G[i1 * cv + o];
    }
    const uint32_t pa[4] = {p0.x, p0.y, p0.z, p0.w}, ga[4] = {g0.x, g0.y, g0.z, g0.w};
    const uint32_t pb[4] = {p1.x, p1.y, p1.z, p1.w}, gb[4] = {g1.x, g1.y, g1.z, g1.w};
    uint32_t *dst = tw + (8 * q) * kGateChW + rl * kGateRowW + sp;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      dst[(2 * w) * kGateChW] = pack_bf16x2(sigmoid_f(bf16_lo(ga[w])) * bf16_lo(pa[w]),
                                            sigmoid_f(bf16_lo(gb[w])) * bf16_lo(pb[w]));
      dst[(2 * w + 1) * kGateChW] = pack_bf16x2(sigmoid_f(bf16_hi(ga[w])) * bf16_hi(pa[w]),
                                                sigmoid_f(bf16_hi(gb[w])) * bf16_hi(pb[w]));
    }
  }
  __syncthreads();
  uint16_t *out = op ? g.out[1] : g.out[0];
#pragma unroll 2
  for (int e = threadIdx.x; e < kGateCG * kGateT * 2; e += kGateThreads) {
    const int half = e & 1, rl = (e >> 1) & 15, cl = e >> 5;
    const int r = r0 + rl, s = s0 + 8 * half;
    if (cl >= 8 * nq || r >= N || s >= N) continue;  // N is a multiple of 8: whole 8-value chunks
    const uint32_t *src = tw + cl * kGateChW + rl * kGateRowW + 4 * half;
    *reinterpret_cast<uint4 *>(out + (((int64_t)b * C + c0 + cl) * N + r) * N + s) =
        make_uint4(src[0], src[1], src[2], src[3]);
  }
}

// ---------------------------------------------------------------- gating gradient: channel-major -> pair
// dP[b,x,y,c] = dA[b,c,r,s] sigmoid(G), dG = dA P sigmoid(G) (1 - sigmoid(G)), (x, y) = (r, s) or
// (s, r): the inverse of the gating kernel's layout change. One CTA: 16 x 16 positions and up to
// 32 channels of one operand. dA rows (c, r) of 16 FP32 values are read with 16-byte loads into
// shared memory [channel][r][s] (channel stride 289 words, row pitch 17); each thread then takes
// 8 channels of one position and writes 16 bytes of dP and of dG. Its P and G chunks are loaded
// before the dA tile, so that both loads' latencies overlap.
constexpr int kGbCG = 32, kGbRowW = 17, kGbChW = 289;
constexpr int kGbSmem = kGbCG * kGbChW * 4;

struct GateBwdArgs {
  const float *dA[2];
  const uint16_t *P[2], *G[2];
  uint16_t *dP[2], *dG[2];
  int N, C, groups, transposed;
};

__global__ void __launch_bounds__(kGateThreads) trimul_gate_bwd_kernel(const GateBwdArgs g) {
  extern __shared__ float tf[];  // [32][289]
  int op, grp, b, r0, s0;
  tile_of(g.N, g.groups, op, grp, b, r0, s0);
  const int N = g.N, C = g.C, c0 = grp * kGbCG, nq = min(kGbCG, C - c0) / 8;
  const float *dA = op ? g.dA[1] : g.dA[0];
  const uint4 *P = reinterpret_cast<const uint4 *>(op ? g.P[1] : g.P[0]),
              *G = reinterpret_cast<const uint4 *>(op ? g.G[1] : g.G[0]);
  uint4 *dP = reinterpret_cast<uint4 *>(op ? g.dP[1] : g.dP[0]), *dG = reinterpret_cast<uint4 *>(op ? g.dG[1] : g.dG[0]);
  const int64_t cv = C / 8;
  // this thread's P and G chunks (8 channels of one position, four positions) are requested
  // first, so that their latency overlaps the dA loads and the barrier
  constexpr int kIt = kGateT * kGateT * 4 / kGateThreads;
  uint4 pv[kIt], gv[kIt];
  int64_t idx[kIt];
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int e = threadIdx.x + it * kGateThreads;
    const int q = e & 3, sl = (e >> 2) & 15, rl = e >> 6;
    const int r = r0 + rl, s = s0 + sl;
    idx[it] = -1;
    if (q < nq && r < N && s < N) {
      const int64_t pos = g.transposed ? ((int64_t)b * N + s) * N + r : ((int64_t)b * N + r) * N + s;
      idx[it] = pos * cv + c0 / 8 + q;
      pv[it] = P[idx[it]];
      gv[it] = G[idx[it]];
    }
  }
#pragma unroll
  for (int e = threadIdx.x; e < kGbCG * kGateT * 4; e += kGateThreads) {
    const int qt = e & 3, rl = (e >> 2) & 15, cl = e >> 6;
    const int r = r0 + rl, s = s0 + 4 * qt;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (cl < 8 * nq && r < N && s < N)  // N is a multiple of 8: whole 4-value chunks
      v = *reinterpret_cast<const float4 *>(dA + (((int64_t)b * C + c0 + cl) * N + r) * N + s);
    float *dst = tf + cl * kGbChW + rl * kGbRowW + 4 * qt;
    dst[0] = v.x, dst[1] = v.y, dst[2] = v.z, dst[3] = v.w;
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    if (idx[it] < 0) continue;
    const int e = threadIdx.x + it * kGateThreads;
    const int q = e & 3, sl = (e >> 2) & 15, rl = e >> 6;
    const uint32_t pw[4] = {pv[it].x, pv[it].y, pv[it].z, pv[it].w}, gw[4] = {gv[it].x, gv[it].y, gv[it].z, gv[it].w};
    const float *src = tf + (8 * q) * kGbChW + rl * kGbRowW + sl;
    uint32_t op_[4], og[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float d0 = src[(2 * w) * kGbChW], d1 = src[(2 * w + 1) * kGbChW];
      const float sg0 = sigmoid_f(bf16_lo(gw[w])), sg1 = sigmoid_f(bf16_hi(gw[w]));
      op_[w] = pack_bf16x2(d0 * sg0, d1 * sg1);
      og[w] = pack_bf16x2(d0 * bf16_lo(pw[w]) * (sg0 * (1.f - sg0)), d1 * bf16_hi(pw[w]) * (sg1 * (1.f - sg1)));
    }
    dP[idx[it]] = make_uint4(op_[0], op_[1], op_[2], op_[3]);
    dG[idx[it]] = make_uint4(og[0], og[1], og[2], og[3]);
  }
}

// ---------------------------------------------------------------- gating, channel-major layout
// A = bf16(sigmoid(G) P) element by element when P and G are already channel-major [B, C, N, N]:
// a streaming kernel, 16-byte loads and stores, four chunks of 8 values per thread in flight.
struct GateCmArgs {
  const uint16_t *P[2], *G[2];
  uint16_t *out[2];
  int64_t chunks;  // 8-value chunks per operand
};

__global__ void __launch_bounds__(256) trimul_gate_cm_kernel(const GateCmArgs g) {
  const int op = blockIdx.y;
  const uint4 *P = reinterpret_cast<const uint4 *>(op ? g.P[1] : g.P[0]),
              *G = reinterpret_cast<const uint4 *>(op ? g.G[1] : g.G[0]);
  uint4 *out = reinterpret_cast<uint4 *>(op ? g.out[1] : g.out[0]);
  const int64_t base = (int64_t)blockIdx.x * (256 * 4) + threadIdx.x;
  uint4 pv[4], gv[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t i = base + 256 * k;
    if (i < g.chunks) pv[k] = P[i], gv[k] = G[i];
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t i = base + 256 * k;
    if (i >= g.chunks) continue;
    const uint32_t pw[4] = {pv[k].x, pv[k].y, pv[k].z, pv[k].w}, gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
    uint32_t o[4];
#pragma unroll
    for (int w = 0; w < 4; ++w)
      o[w] = pack_bf16x2(sigmoid_f(bf16_lo(gw[w])) * bf16_lo(pw[w]), sigmoid_f(bf16_hi(gw[w])) * bf16_hi(pw[w]));
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------- batched GEMM D = A B^T
// D[t][m][n] = sum_k Aop[t][m][k] Bop[t][n][k] for a stack of N x N BF16 matrices (t = batch x
// channel), FP32 accumulation in TMEM. Operand storage: K-major = [m][k] (k contiguous), MN-major
// = [k][m] (m contiguous). The epilogue either stores D (row-major [t][m][n], BF16 or FP32) or,
// for the backward pass in the channel-major layout, applies the gating gradient to D = dA on
// the fly: dP = dA sigmoid(G), dG = dA P sigmoid(G) (1 - sigmoid(G)), with P and G read at the
// same [t][m][n] positions.
//
// Persistent CTAs, one per SM, walk the tiles t, m / 128, n / 256 (n fastest). Warp 0 issues the
// TMA loads of a 4-stage ring (K step 64: one 128-byte swizzle atom of the K-major rows, or 64 rows
// of the MN-major ones); warp 1 owns TMEM and issues the tcgen05.mma (M = 128, N = 256, K = 16)
// into one of two accumulators; warps 2-9 (two per TMEM lane quarter, one per half of the
// columns) read the other accumulator out, so the epilogue of one tile overlaps the main loop of
// the next.
enum { kEpiBF16 = 0, kEpiF32 = 1, kEpiGate = 2 };

struct GemmIO {
  void *D;                // kEpiBF16 / kEpiF32: the product
  const uint16_t *P, *G;  // kEpiGate: projection and gate logits of the gated operand, D's layout
  uint16_t *dP, *dG;      // kEpiGate: their gradients
};

struct GemmCfg {
  static constexpr int BM = 128, BN = 256, BK = 64, NST = 4;
  static constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE = A_BYTES + B_BYTES;
  static constexpr int MN_BOX = BK * 128;  // bytes of one 64-wide MN-major box (BK rows of 128 bytes)
  static constexpr int EPI_WARPS = 8;                  // a multiple of 4: whole TMEM lane quarters
  static constexpr int EPI_CPW = BN / 32 / (EPI_WARPS / 4);  // 32-column chunks per epilogue warp
  static constexpr int EPI_PITCH = 33;                 // words per row of a warp's 32 x 32 staging tile
  static constexpr int EPI_TILE = 32 * EPI_PITCH * 4;  // bytes
  static constexpr int OFF_EPI = NST * STAGE;
  static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_TILE;
  static constexpr int B_FULL = 0, B_EMPTY = NST, B_ACCF = 2 * NST, B_ACCE = B_ACCF + 2, B_DONE = B_ACCE + 2,
                       NBAR = B_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 64 + 32 * EPI_WARPS;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(STAGE % 1024 == 0 && A_BYTES % 1024 == 0, "SW128 tiles need 1 KB alignment");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Stores 8 consecutive values v of one row of D at element offset `off` (the epilogue's unit of
// work after the staging transpose): FP32, BF16, or the gating gradient from P and G (pv, gv).
template <int kEpi>
__device__ __forceinline__ void gemm_store8(const GemmIO &io, int64_t off, const float (&v)[8], const uint4 &pv,
                                            const uint4 &gv) {
  if constexpr (kEpi == kEpiF32) {
    float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(io.D) + off);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else if constexpr (kEpi == kEpiBF16) {
    *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(io.D) + off) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  } else {
    const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t op_[4], og[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float d0 = v[2 * x], d1 = v[2 * x + 1];
      const float s0 = sigmoid_f(bf16_lo(gw[x])), s1 = sigmoid_f(bf16_hi(gw[x]));
      op_[x] = pack_bf16x2(d0 * s0, d1 * s1);
      og[x] = pack_bf16x2(d0 * bf16_lo(pw[x]) * (s0 * (1.f - s0)), d1 * bf16_hi(pw[x]) * (s1 * (1.f - s1)));
    }
    *reinterpret_cast<uint4 *>(io.dP + off) = make_uint4(op_[0], op_[1], op_[2], op_[3]);
    *reinterpret_cast<uint4 *>(io.dG + off) = make_uint4(og[0], og[1], og[2], og[3]);
  }
}

template <bool kAMN, bool kBMN, int kEpi>
__global__ void __launch_bounds__(GemmCfg::NTHREADS, 1)
    trimul_gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                       const GemmIO io, int N, int batch, int *status) {
  using C = GemmCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int k) { return sb0 + C::OFF_BAR + 8u * (uint32_t)k; };
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_MISC);
  const Abort ab{reinterpret_cast<volatile int *>(misc + 1), status};
  const int mt = (N + C::BM - 1) / C::BM, nt = (N + C::BN - 1) / C::BN, nk = (N + C::BK - 1) / C::BK;
  const int ntiles = batch * mt * nt;
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
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    bool ok = true;
    int it = 0;
    if (lane == 0) {
      tma_prefetch_map(&mA);
      tma_prefetch_map(&mB);
    }
    for (int u = blockIdx.x; u < ntiles && ok; u += gridDim.x) {
      int t, m0, n0;
      tile_of(u, t, m0, n0);
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int st = it % C::NST;
        if (it >= C::NST) ok = wait_bar_warp(bar(C::B_EMPTY + st), ((it / C::NST) - 1) & 1, ab);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t dst = sb0 + st * C::STAGE, fb = bar(C::B_FULL + st);
          const int k0 = kb * C::BK;
          mbar_arrive_expect_tx(fb, C::STAGE);
          if constexpr (kAMN) {
#pragma unroll
            for (int x = 0; x < C::BM / 64; ++x) tma_load_3d(dst + x * C::MN_BOX, &mA, fb, m0 + 64 * x, k0, t);
          } else {
            tma_load_3d(dst, &mA, fb, k0, m0, t);
          }
          if constexpr (kBMN) {
#pragma unroll
            for (int x = 0; x < C::BN / 64; ++x)
              tma_load_3d(dst + C::A_BYTES + x * C::MN_BOX, &mB, fb, n0 + 64 * x, k0, t);
          } else {
            tma_load_3d(dst + C::A_BYTES, &mB, fb, k0, n0, t);
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
    // K step of 16 within a stage: 32 bytes along a K-major swizzled row, or 16 rows (2 KB) of an
    // MN-major tile; descriptors count 16-byte units
    constexpr uint64_t a_step = kAMN ? (16 * 128) >> 4 : 32 >> 4;
    constexpr uint64_t b_step = kBMN ? (16 * 128) >> 4 : 32 >> 4;
    bool ok = true;
    int it = 0, tl = 0;
    for (int u = blockIdx.x; u < ntiles && ok; u += gridDim.x, ++tl) {
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
        // MN-major: leading offset = stride between 64-element MN blocks, stride offset = 8 K rows
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
    // every MMA issued so far has completed once this commit arrives: TMEM can be released
    mma_commit_e(bar(C::B_DONE));
    if (lane == 0) drain_bar(bar(C::B_DONE), 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue: TMEM -> registers -> global
    // Per 32 x 32 chunk: TMEM rows (one per thread) go through the warp's staging tile, then every
    // thread takes 8-value pieces of four rows, so that one warp instruction covers 8 rows of 32
    // contiguous values (conflict-free: pitch 33 words).
    const int q = warp & 3;                             // the TMEM lane quarter this warp may access
    const int cbase = ((warp - 2) >> 2) * (32 * C::EPI_CPW);  // its share of the columns
    const uint32_t lrow = (uint32_t)(q * 32) << 16;
    float *stg = reinterpret_cast<float *>(sm + C::OFF_EPI + (warp - 2) * C::EPI_TILE);
    const int rq = lane >> 2, cq = lane & 3;
    int tl = 0;
    for (int u = blockIdx.x; u < ntiles; u += gridDim.x, ++tl) {
      int t, m0, n0;
      tile_of(u, t, m0, n0);
      const int acc = tl & 1;
      if (!wait_bar_warp(bar(C::B_ACCF + acc), (tl >> 1) & 1, ab)) break;
      tc_fence_after();
      const int mrow = m0 + q * 32 + rq;  // this thread's rows: mrow + 8 i
      // P and G of the next chunk are requested before the current one is processed (two sets in
      // flight per thread)
      uint4 pv[2][4], gv[2][4];
      auto load_pg = [&](int c0, uint4(&p)[4], uint4(&g)[4]) {
        const int col = n0 + c0 + 8 * cq;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (mrow + 8 * i < N && col < N) {
            const int64_t off = ((int64_t)t * N + mrow + 8 * i) * N + col;
            p[i] = *reinterpret_cast<const uint4 *>(io.P + off);
            g[i] = *reinterpret_cast<const uint4 *>(io.G + off);
          }
      };
      if constexpr (kEpi == kEpiGate) load_pg(cbase, pv[0], gv[0]);
#pragma unroll
      for (int k = 0; k < C::EPI_CPW; ++k) {  // this warp's 32-column chunks
        const int c0 = cbase + 32 * k, n = n0 + c0;
        if (n >= N) break;  // uniform across the warp
        if constexpr (kEpi == kEpiGate)
          if (k + 1 < C::EPI_CPW && n + 32 < N) load_pg(c0 + 32, pv[(k + 1) & 1], gv[(k + 1) & 1]);
        const int col = n + 8 * cq;
        uint32_t r[32];
        tmem_ld32(tb + lrow + acc * C::BN + c0, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) stg[lane * C::EPI_PITCH + j] = __uint_as_float(r[j]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = stg[(rq + 8 * i) * C::EPI_PITCH + 8 * cq + j];
          if (mrow + 8 * i < N && col < N)  // N is a multiple of 8: whole 8-value pieces
            gemm_store8<kEpi>(io, ((int64_t)t * N + mrow + 8 * i) * N + col, v, pv[k & 1][i], gv[k & 1][i]);
        }
        __syncwarp();  // the staging tile is rewritten by the next chunk
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_ACCE + acc));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
// 3-D TMA view (inner, outer, t) of a BF16 stack of N x N matrices; one box is 64 inner elements
// (128 bytes, 128-byte swizzled) x `rows` outer rows. Elements past N read as zeros.
cudaError_t make_stack_map(CUtensorMap *m, const void *ptr, int N, int batch, int rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)batch};
  cuuint64_t strides[2] = {2ull * N, 2ull * N * N};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool kAMN, bool kBMN, int kEpi>
struct Gemm {
  CUtensorMap mA, mB;
  int grid;
  // Tensor maps and one-time attribute set-up; nothing is launched.
  cudaError_t plan(const uint16_t *A, const uint16_t *B, int N, int batch) {
    cudaError_t e = make_stack_map(&mA, A, N, batch, kAMN ? GemmCfg::BK : GemmCfg::BM);
    if (e == cudaSuccess) e = make_stack_map(&mB, B, N, batch, kBMN ? GemmCfg::BK : GemmCfg::BN);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    e = current_device(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    static DeviceOnce ready;
    if (!ready.done(dev)) {
      e = cudaFuncSetAttribute(trimul_gemm_kernel<kAMN, kBMN, kEpi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               GemmCfg::SMEM_ALLOC);
      if (e != cudaSuccess) return e;
      ready.mark(dev);
    }
    const int64_t tiles =
        (int64_t)batch * ((N + GemmCfg::BM - 1) / GemmCfg::BM) * ((N + GemmCfg::BN - 1) / GemmCfg::BN);
    grid = (int)std::min<int64_t>(tiles, nsm);
    return cudaSuccess;
  }
  cudaError_t launch(const GemmIO &io, int N, int batch, int *status, cudaStream_t st) const {
    trimul_gemm_kernel<kAMN, kBMN, kEpi>
        <<<grid, GemmCfg::NTHREADS, GemmCfg::SMEM_ALLOC, st>>>(mA, mB, io, N, batch, status);
    return cudaGetLastError();
  }
};

cudaError_t gate_setup() {
  int dev = 0;
  cudaError_t e = current_device(&dev);
  if (e != cudaSuccess) return e;
  static DeviceOnce ready;
  if (!ready.done(dev)) {
    e = cudaFuncSetAttribute(trimul_gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGateSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(trimul_gate_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGbSmem);
    if (e != cudaSuccess) return e;
    ready.mark(dev);
  }
  return cudaSuccess;
}

int check_shape(const tri_mul_shape &s) {
  if (s.B < 1 || s.N < 1 || s.C < 1 || (s.incoming != 0 && s.incoming != 1) ||
      (s.layout != TRI_MUL_LAYOUT_PAIR && s.layout != TRI_MUL_LAYOUT_CHANNEL_MAJOR))
    return TRI_ATTN_ERR_INVALID_ARG;
  if (s.N < 16 || s.N > TRI_MUL_MAX_N || s.N % 8 || s.C < 8 || s.C > TRI_MUL_MAX_C || s.C % 8 ||
      (int64_t)s.B * s.C > 65535)
    return TRI_ATTN_ERR_UNSUPPORTED;
  return TRI_ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t stack_elems(const tri_mul_shape &s) { return (size_t)s.B * s.C * (size_t)s.N * s.N; }

// Channel-major backward: both products with the gating gradient fused into their epilogues.
// Outgoing (X = A Bm^T): dA = dX Bm (dX K-major, Bm MN-major), dB = dX^T A (both MN-major).
// Incoming (X = A^T Bm, operands stored [k][i]): dA[k][i] = sum_j Bm[k][j] dX[i][j] (both K-major),
// dB[k][j] = sum_i A[k][i] dX[i][j] (A K-major, dX MN-major).
template <bool kA1, bool kB1, bool kA2, bool kB2>
int mul_bwd_cm(const tri_mul_shape &s, const uint16_t *Pa, const uint16_t *Ga, const uint16_t *Pb, const uint16_t *Gb,
               const uint16_t *A, const uint16_t *Bm, const uint16_t *dX, uint16_t *dPa, uint16_t *dGa, uint16_t *dPb,
               uint16_t *dGb, int *status, cudaStream_t st) {
  const int N = s.N, T = s.B * s.C;
  Gemm<kA1, kB1, kEpiGate> ga_;
  Gemm<kA2, kB2, kEpiGate> gb_;
  const uint16_t *a1 = s.incoming ? Bm : dX, *b1 = s.incoming ? dX : Bm;
  const uint16_t *a2 = s.incoming ? A : dX, *b2 = s.incoming ? dX : A;
  if (ga_.plan(a1, b1, N, T) != cudaSuccess || gb_.plan(a2, b2, N, T) != cudaSuccess)
    return TRI_ATTN_ERR_CUDA;
  cudaError_t e = ga_.launch(GemmIO{nullptr, Pa, Ga, dPa, dGa}, N, T, status, st);
  if (e == cudaSuccess) e = timing_mark(0, st);
  if (e == cudaSuccess) e = gb_.launch(GemmIO{nullptr, Pb, Gb, dPb, dGb}, N, T, status, st);
  if (e == cudaSuccess) e = timing_mark(1, st);
  return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA;
}

}  // namespace

}  // namespace triattn

using namespace triattn;

extern "C" {

int tri_mul_fwd(tri_mul_shape shape, const tri_attn_bf16 *Pa, const tri_attn_bf16 *Ga, const tri_attn_bf16 *Pb,
                const tri_attn_bf16 *Gb, tri_attn_bf16 *A, tri_attn_bf16 *Bm, tri_attn_bf16 *X, void *stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  const void *ptrs[] = {Pa, Ga, Pb, Gb, A, Bm, X};
  for (const void *p : ptrs) {
    if (!p) return TRI_ATTN_ERR_INVALID_ARG;
    if (!aligned16(p)) return TRI_ATTN_ERR_UNSUPPORTED;
  }
  const int N = shape.N, T = shape.B * shape.C;
  int *status = device_status_word();
  if (!status) return TRI_ATTN_ERR_CUDA;
  auto st = static_cast<cudaStream_t>(stream);
  const bool cm = shape.layout == TRI_MUL_LAYOUT_CHANNEL_MAJOR;
  // the pair layout's gating transposes the incoming operands, so its contraction is always
  // X = A Bm^T; the channel-major layout keeps them as stored and reads them MN-major instead
  Gemm<false, false, kEpiBF16> g_out;
  Gemm<true, true, kEpiBF16> g_in;
  const bool mn = cm && shape.incoming;
  if ((mn ? g_in.plan(A, Bm, N, T) : g_out.plan(A, Bm, N, T)) != cudaSuccess || gate_setup() != cudaSuccess)
    return TRI_ATTN_ERR_CUDA;
  cudaError_t e;
  if (cm) {
    GateCmArgs ga{{Pa, Pb}, {Ga, Gb}, {A, Bm}, (int64_t)(stack_elems(shape) / 8)};
    const dim3 grid((unsigned)((ga.chunks + 1023) / 1024), 2);
    trimul_gate_cm_kernel<<<grid, 256, 0, st>>>(ga);
  } else {
    GateArgs ga{{Pa, Pb}, {Ga, Gb}, {A, Bm}, N, shape.C, (shape.C + kGateCG - 1) / kGateCG, shape.incoming};
    const int nt = (N + kGateT - 1) / kGateT;
    trimul_gate_kernel<<<shape.B * nt * nt * ga.groups * 2, kGateThreads, kGateSmem, st>>>(ga);
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) e = timing_mark(0, st);
  const GemmIO io{X, nullptr, nullptr, nullptr, nullptr};
  if (e == cudaSuccess) e = mn ? g_in.launch(io, N, T, status, st) : g_out.launch(io, N, T, status, st);
  if (e == cudaSuccess) e = timing_mark(1, st);
  return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA;
}

size_t tri_mul_bwd_workspace_size(tri_mul_shape shape) {
  if (check_shape(shape)) return 0;
  return shape.layout == TRI_MUL_LAYOUT_CHANNEL_MAJOR ? 0 : 2 * sizeof(float) * stack_elems(shape);
}

int tri_mul_bwd(tri_mul_shape shape, const tri_attn_bf16 *Pa, const tri_attn_bf16 *Ga, const tri_attn_bf16 *Pb,
                const tri_attn_bf16 *Gb, const tri_attn_bf16 *A, const tri_attn_bf16 *Bm, const tri_attn_bf16 *dX,
                tri_attn_bf16 *dPa, tri_attn_bf16 *dGa, tri_attn_bf16 *dPb, tri_attn_bf16 *dGb, void *workspace,
                size_t workspace_bytes, void *stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  const void *ptrs[] = {Pa, Ga, Pb, Gb, A, Bm, dX, dPa, dGa, dPb, dGb};
  for (const void *p : ptrs) {
    if (!p) return TRI_ATTN_ERR_INVALID_ARG;
    if (!aligned16(p)) return TRI_ATTN_ERR_UNSUPPORTED;
  }
  if (workspace && !aligned16(workspace)) return TRI_ATTN_ERR_UNSUPPORTED;
  const size_t need = tri_mul_bwd_workspace_size(shape);
  if (need && (!workspace || workspace_bytes < need)) return TRI_ATTN_ERR_WORKSPACE;
  int *status = device_status_word();
  if (!status) return TRI_ATTN_ERR_CUDA;
  auto st = static_cast<cudaStream_t>(stream);
  if (shape.layout == TRI_MUL_LAYOUT_CHANNEL_MAJOR)
    return shape.incoming ? mul_bwd_cm<false, false, false, true>(shape, Pa, Ga, Pb, Gb, A, Bm, dX, dPa, dGa, dPb,
                                                                  dGb, status, st)
                          : mul_bwd_cm<false, true, true, true>(shape, Pa, Ga, Pb, Gb, A, Bm, dX, dPa, dGa, dPb,
                                                                dGb, status, st);
  const int N = shape.N, T = shape.B * shape.C;
  float *dA = static_cast<float *>(workspace);
  float *dB = dA + stack_elems(shape);
  // pair layout: dA[t] = dX[t] Bm[t] (Bm read MN-major) and dB[t] = dX[t]^T A[t] (both operands
  // MN-major) in FP32, then the gating gradient maps them back to the pair layout
  Gemm<false, true, kEpiF32> gemm_a;
  Gemm<true, true, kEpiF32> gemm_b;
  if (gemm_a.plan(dX, Bm, N, T) != cudaSuccess || gemm_b.plan(dX, A, N, T) != cudaSuccess ||
      gate_setup() != cudaSuccess)
    return TRI_ATTN_ERR_CUDA;
  cudaError_t e = gemm_a.launch(GemmIO{dA, nullptr, nullptr, nullptr, nullptr}, N, T, status, st);
  if (e == cudaSuccess) e = timing_mark(0, st);
  if (e == cudaSuccess) e = gemm_b.launch(GemmIO{dB, nullptr, nullptr, nullptr, nullptr}, N, T, status, st);
  if (e == cudaSuccess) e = timing_mark(1, st);
  if (e == cudaSuccess) {
    GateBwdArgs gg{{dA, dB}, {Pa, Pb}, {Ga, Gb}, {dPa, dPb}, {dGa, dGb}, N, shape.C,
                   (shape.C + kGbCG - 1) / kGbCG, shape.incoming};
    const int nt = (N + kGateT - 1) / kGateT;
    trimul_gate_bwd_kernel<<<shape.B * nt * nt * gg.groups * 2, kGateThreads, kGbSmem, st>>>(gg);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = timing_mark(2, st);
  return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA;
}

}  // extern "C"
