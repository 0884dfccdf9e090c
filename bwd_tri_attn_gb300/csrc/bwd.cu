// Backward pass: key-tile-parallel tcgen05 kernel that recomputes every
// probability tile exactly once and produces dQ, dK, dV and the dBias partials.
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract): the shared pair bias adds a
// reduction over slices to the usual reductions over queries (dK, dV) and keys
// (dQ); the key-tile-parallel backward recomputes each probability tile once
// and uses ordered partial reductions, with no floating-point atomics and no
// full score-gradient storage.
//
// Work unit (one CTA): key tile kt (128 keys) of a contiguous range of (head, slice) pairs (the
// range of the CTA's cluster, below), walked head by head in blocks of GB slices:
//     for block: for query tile jt: for slice i in block:     (one "step")
//         S^T  = K_i Q_i[jt]^T        (TMEM, lanes = keys)
//         dP^T = V_i dO_i[jt]^T
//         P^T  = exp2(S^T*scale*log2e + biasT*log2e - LSE*log2e)   (FP32, written back as FP16)
//         dS^T = P^T * (dP^T - D)      (P rounded to FP16 first: it is also the dV operand)
//         dV_i += P^T dO_i[jt],  dK_i += dS^T Q_i[jt]            (TMEM accumulators, one pair per slice of the block)
//         dQ_i[jt] partial = dS K_i                               (reduced across the cluster, below)
//         dBias tile (jt, kt) += dS   (registers, summed in slice order over the block)
//     after each (block, jt): the dBias tile is added into the cluster's FP32 partial slot for the head
//     (this CTA owns the tile)
//     after each block: dK_i, dV_i -> BF16
//
// Three reductions, each in a fixed order:
//  - dK, dV over query tiles: in the CTA's TMEM accumulator, jt = 0, 1, ...
//  - dQ over key tiles: the n = N/128 CTAs of one key-tile row form a
//    thread-block cluster. CTA r owns query rows [r*128/n, (r+1)*128/n) of every
//    step's tile; each CTA pushes the matching rows of its 128 x d FP32 partial
//    into the owner's receive buffer with st.async (completing bytes on the
//    owner's mbarrier), and the owner sums the n partials in rank (= kt) order,
//    one step later so that the exchange overlaps the next step's work. The
//    receive buffer has two slots used by alternate steps, so a CTA can push step
//    t while an owner is still summing step t - 1.
//  - dBias over slices: within a block in slice order (registers), across blocks in
//    block order (the partial slot), across the slots of a head in slot order (reduce kernel).
// Every order depends on the shape and the number of resident clusters (the GPU model) only.
//
// Operands: all tensor-core operands are FP16; P and dS need FP16's 11-bit significand. Q, K,
// V and dO are converted in shared memory after multiplication by the power of two of their
// (batch, head) block (exponents from the preparation kernel: sq, sk, sv, so), which keeps every
// entry within 2^-20 of the block's largest one exact in FP16. The scales are undone exactly and
// change only between heads, so every role sets its constants once per block of slices: S^T
// carries 2^(sk+sq) (folded into the exponent's scale factor), dP^T carries w = 2^(sv+so), so
// dS' = P (dP^T - w D) is w times the unscaled FP32 dS to the bit and is packed to FP16 as it
// stands (|dS'| < 2^14 by the choice of sv, so); the dBias register sums carry w (removed with
// one FFMA per element at the flush), dK carries w 2^sq, dV 2^so and the dQ partials w 2^sk
// (removed by the owner after it has summed them), all in FP32 before the BF16 rounding.
//
// Warp roles (8 + NEW warps; NEW = 8 with QPT = 64 queries per elementwise thread). The control
// warps take the lowest indices (warp schedulers favour low-index warps, and their short
// instruction sequences gate everyone else's progress):
//   0         TMA producer (+ LSE / D rows), 1 MMA issuer and TMEM owner, 2..3 BF16 -> FP16 conversion
//   4..7      dQ: read the dQ partial from TMEM (lanes = queries), push it to the owners, reduce owned rows
//   8..8+NEW-1 elementwise: thread = key row (TMEM lane quarter w % 4) x QPT queries (column group (w - 8) / 4);
//             only P and dS are on their path; the most registers (setmaxnreg)
// TMEM columns: A = [0,128) S^T, then FP16 P^T; B = [128,256) dP^T, then FP16 dS^T; dK_i, dV_i
// from 256. Each elementwise thread writes P^T (dS^T) as packed FP16 over the S^T (dP^T) columns
// it has just read: column group g of 64 queries keeps its 32 packed columns at A + 64g (B + 64g).
// The dQ partial (128 queries x d, FP32) takes B + [32, 64), which dS^T leaves free. dV = P^T dO
// is issued as soon as the P phase is done and S^T(t+1) right behind it: the MMAs of one issuing
// thread are performed in issue order, so S^T(t+1) cannot overwrite region A before dV(t) has
// read it. dK = dS^T Q follows the dS phase, and dP^T(t+1) follows dK(t) into region B once the
// dQ warps have read dQ(t) out of B (their tcgen05.ld is the one wait this needs); dQ = dS K reads
// dS from a 128-byte-swizzled FP16 tile in shared memory. So the P phase of step t+1 overlaps
// step t's dK and dQ. A new block of slices waits for dV(t) to complete before its S^T, since
// it needs the block's new K and V in shared memory.
#include "common.cuh"
#include "launch.cuh"
#include "plan.cuh"
#include "sm100.cuh"
#include "sync.cuh"
#include "tmap.cuh"

namespace triattn {
using namespace sm100;

template <int HD>
struct BwdCfg {
  static constexpr int GB = HD == 32 ? 4 : 8;  // slices per block: dK/dV of GB slices live in TMEM
  static constexpr int NQS = 3;                // Q/dO stages
  static constexpr int ROWB = HD * 2;
  static constexpr int TILE = 128 * ROWB;
  static constexpr uint32_t SW = HD == 32 ? kSwizzle64B : kSwizzle32B;
  static constexpr int QPT = 64;                   // queries per elementwise thread (64: 8 warps, 32: 16)
  static constexpr int NEW = 4 * 128 / QPT, NEWT = NEW * 32;  // elementwise warps WARP_EW0 .. WARP_EW0 + NEW - 1
  static constexpr int KPG = QPT / 16;             // K steps of 16 queries per column group
  static constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CV = 2, NCV = 2, NCVT = NCV * 32;
  static constexpr int WARP_DQ = 4, NDQ = 4, NDQT = NDQ * 32, WARP_EW0 = 8;
  static constexpr int NTHREADS = (NEW + 8) * 32;
  static constexpr uint32_t REG_LAUNCH = QPT == 64 ? 128 : 80, REG_EW = QPT == 64 ? 200 : 96,
                            REG_OTHER = 48, REG_DQ = 64;
  // warpgroup 0 (producer, MMA issuer, converters) keeps REG_OTHER, warpgroup 1 (dQ) REG_DQ
  static_assert(NEWT * REG_EW + 128 * REG_OTHER + 128 * REG_DQ == NTHREADS * REG_LAUNCH, "register split");
  // the dQ partial (32 columns) uses the half of region B that dS^T leaves free: column group 0 of
  // the elementwise threads keeps its packed dS^T in B + [0,32) and group 1 in B + [64,96)
  static constexpr uint32_t TA = 0, TB = 128, TDQ = TB + 32, TDKV = 256, TMEM_COLS = 512;
  static_assert(QPT == 64 && HD <= 32, "dQ partial inside region B");
  static_assert(TDKV + GB * 2 * HD <= TMEM_COLS, "TMEM budget");
  static constexpr int BIAS_TILE = 128 * 128 * 2;
  static constexpr int RB_ROWS = 136;  // >= n * ceil(128 / n) for every cluster size n <= 8
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + GB * TILE;
  static constexpr int OFF_Q = OFF_V + GB * TILE;
  static constexpr int OFF_DO = OFF_Q + NQS * TILE;
  static constexpr int OFF_BIAS = OFF_DO + NQS * TILE;     // [2 halves][128 rows][128 B], SW128
  static constexpr int OFF_DS = OFF_BIAS + BIAS_TILE;      // FP16 dS, MN-major SW128: [16 key groups][2][8][128 B]
  static constexpr int RB_SLOT = RB_ROWS * HD * 4;
  static constexpr int NRB = 2;                            // dQ receive slots (step t uses slot t % NRB)
  static constexpr int OFF_RB = OFF_DS + 32768;            // dQ receive buffers: NRB x [sender][row][HD] FP32
  static constexpr int OFF_LSE = OFF_RB + NRB * RB_SLOT;   // [NQS][128]: -LSE*log2e (or -inf)
  static constexpr int OFF_D = OFF_LSE + NQS * 512;          // [NQS][128]: D
  static constexpr int OFF_MASK = OFF_D + NQS * 512;         // [GB][128]: mask*log2e of this CTA's keys
  static constexpr int OFF_DQF = OFF_MASK + GB * 512;        // [NDQ warps][2 blocks][2] float: dQ factors
  static constexpr int OFF_BAR = OFF_DQF + NDQ * 16;
  static constexpr int B_KVFULL = 0, B_KVREADY = 1, B_KVFREE = 2;
  static constexpr int B_QDOFULL = 3, B_QDOREADY = B_QDOFULL + NQS, B_QDOFREE = B_QDOREADY + NQS;
  static constexpr int B_BFULL = B_QDOFREE + NQS, B_BFREE = B_BFULL + 1;  // the (single) bias tile
  static constexpr int B_SFULL = B_BFREE + 1, B_PAFULL = B_SFULL + 1, B_AFREE = B_PAFULL + 1;
  static constexpr int B_DPFULL = B_AFREE + 1, B_PFULL = B_DPFULL + 1;
  static constexpr int B_M2DONE = B_PFULL + 1, B_DQREAD = B_M2DONE + 1;
  static constexpr int B_DKVREAD = B_DQREAD + 1, B_RFULL = B_DKVREAD + 1, B_XEMPTY = B_RFULL + NRB;
  static constexpr int B_FINAL = B_XEMPTY + NRB, NBAR = B_FINAL + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static_assert(OFF_BIAS % 1024 == 0 && OFF_DS % 1024 == 0, "SW128 tiles need 1 KB alignment");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool wait_bar_cluster_warp(uint32_t bar, uint32_t parity, const Abort &ab) {
  const bool ok = wait_bar_cluster(bar, parity, ab);
  return __all_sync(0xffffffffu, ok);
}

// BF16 -> FP16 in place over `bytes` of shared memory, the values multiplied by f (a power of
// two), split across `nthr` threads.
__device__ __forceinline__ void convert_to_f16(uint8_t *p, int bytes, float f, int tid, int nthr) {
  uint4 *v = reinterpret_cast<uint4 *>(p);
  const float2 f2 = make_float2(f, f);
  for (int e = tid; e < bytes / 16; e += nthr) {
    uint4 w = v[e];
    w.x = bf16x2_to_f16x2_scaled2(w.x, f2);
    w.y = bf16x2_to_f16x2_scaled2(w.y, f2);
    w.z = bf16x2_to_f16x2_scaled2(w.z, f2);
    w.w = bf16x2_to_f16x2_scaled2(w.w, f2);
    v[e] = w;
  }
}

// The power-of-two operand scales of one (batch, head) block, from the exponent maxima the
// preparation kernel accumulated (emax[4 hd + {0,1,2,3}] for Q, K, V, dO).
struct BwdScales {
  int sq, sk, sv, so;
};
template <int HD>
__device__ __forceinline__ BwdScales load_scales(const int *emax, int hd) {
  using T = BwdTargets<HD>;
  const int4 e = *reinterpret_cast<const int4 *>(emax + 4 * (int64_t)hd);
  return BwdScales{scale_exp(e.x, kTargetQK), scale_exp(e.y, kTargetQK), scale_exp(e.z, T::TV),
                   scale_exp(e.w, T::TO)};
}


// Work split: the B*H*S (head, slice) pairs, ordered head-major (unit x = head * S + slice,
// head = b * H + h), are cut into NC contiguous ranges, one per cluster: cluster c takes
// [bwd_unit_start(c), bwd_unit_start(c + 1)). NC is as many clusters as the device runs at once,
// so every resident cluster has about the same work. A range may cross head boundaries.
__host__ __device__ inline int bwd_unit_start(int c, int NC, int64_t W) { return (int)((int64_t)c * W / NC); }
// The cluster whose range holds unit x.
__host__ __device__ inline int bwd_cluster_of(int64_t x, int NC, int64_t W) {
  int c = (int)(x * NC / W);
  while (c + 1 < NC && bwd_unit_start(c + 1, NC, W) <= x) ++c;
  while (c > 0 && bwd_unit_start(c, NC, W) > x) --c;
  return c;
}

// The step schedule every role walks in the same order: the CTA's range is cut at head boundaries
// into segments, each segment into blocks of GB slices (the first block of a segment holds f <= GB
// slices, f set per cluster so that clusters reach their dBias flushes at different steps), each
// block into steps: query tiles, then the slices of the block.
struct Sched {
  int beg, end, S, GB, f;
  __device__ static int seg_blocks(int len, int f, int GB) {
    return len <= 0 ? 0 : (len <= f ? 1 : 1 + (len - f + GB - 1) / GB);
  }
  __device__ int nblk() const {
    int n = 0;
    for (int x = beg; x < end;) {
      const int e = min(end, (x / S + 1) * S);
      n += seg_blocks(e - x, f, GB);
      x = e;
    }
    return n;
  }
  // block bi: head, first slice, number of slices, and whether it opens its segment
  __device__ void block(int bi, int &hd, int &i0, int &nb, bool &first) const {
    for (int x = beg; x < end;) {
      const int hx = x / S, e = min(end, (hx + 1) * S), n = seg_blocks(e - x, f, GB);
      if (bi < n) {
        const int off = bi == 0 ? 0 : f + (bi - 1) * GB;
        hd = hx;
        i0 = x - hx * S + off;
        nb = min(bi == 0 ? f : GB, e - x - off);
        first = bi == 0;
        return;
      }
      bi -= n;
      x = e;
    }
    hd = 0;
    i0 = 0;
    nb = 0;
    first = true;
  }
};

template <int HD, int NODE>
__global__ void __launch_bounds__(BwdCfg<HD>::NTHREADS, 1)
bwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
           const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mDO,
           const __grid_constant__ CUtensorMap mBT, const __grid_constant__ CUtensorMap mDK,
           const __grid_constant__ CUtensorMap mDV, const Dims g, const int NC, const int KMAX,
           const float *__restrict__ LSE,
           const float *__restrict__ Dv, const int *__restrict__ emax, const uint16_t *__restrict__ mask,
           uint16_t *__restrict__ dQ, uint16_t *__restrict__ dK, uint16_t *__restrict__ dV,
           float *__restrict__ partial, int *status) {
  using C = BwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkt = (g.N + 127) / 128, njt = nkt;
  const int kt = blockIdx.x, cl = blockIdx.y;  // key tile = cluster rank, cluster index
  const uint32_t rank = cluster_ctarank();     // == kt (the cluster spans the key tiles)
  const int64_t W = (int64_t)g.B * g.H * g.S;
  const Sched sc{bwd_unit_start(cl, NC, W), bwd_unit_start(cl + 1, NC, W), g.S, C::GB, C::GB - cl % C::GB};
  const int nblk = sc.nblk();
  const int T = njt * (sc.end - sc.beg);  // steps of this CTA
  auto bar = [&](int k) { return sb0 + C::OFF_BAR + 8u * (uint32_t)k; };
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_MISC);
  const Abort ab{reinterpret_cast<volatile int *>(misc + 1), status};
  const int r0 = (int)(rank * 128 / nkt), r1 = (int)((rank + 1) * 128 / nkt);  // owned dQ rows
  const int rows_max = (128 + nkt - 1) / nkt;

  if (tid == 0) {
    mbar_init(bar(C::B_KVFULL), 1);
    mbar_init(bar(C::B_KVREADY), C::NCV + C::NEW);  // converter and elementwise warps share the K/V conversion
    mbar_init(bar(C::B_KVFREE), 1);
    for (int s = 0; s < C::NQS; ++s) {
      mbar_init(bar(C::B_QDOFULL + s), 1);
      mbar_init(bar(C::B_QDOREADY + s), C::NCV);
      mbar_init(bar(C::B_QDOFREE + s), 1);
    }
    mbar_init(bar(C::B_BFULL), 1);
    mbar_init(bar(C::B_BFREE), C::NEWT);
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_PAFULL), C::NEWT);
    mbar_init(bar(C::B_AFREE), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PFULL), C::NEWT);
    mbar_init(bar(C::B_M2DONE), 1);
    mbar_init(bar(C::B_DQREAD), C::NDQT);
    mbar_init(bar(C::B_DKVREAD), C::NEWT);
    for (int s = 0; s < C::NRB; ++s) {
      mbar_init(bar(C::B_RFULL + s), 1);             // + the bytes pushed by all n senders
      mbar_init(bar(C::B_XEMPTY + s), C::NDQ * nkt);  // one arrive per dQ warp of every owner
    }
    mbar_init(bar(C::B_FINAL), 1);
    misc[1] = 0;
    fence_barrier_init();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(sb0 + C::OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any peer arrives on them
  tc_fence_after();
  const uint32_t tb = misc[0];
  // Register split (setmaxnreg, per warpgroup, at the top of each warpgroup's branch):
  // warpgroups 0 and 1 give registers up, the two elementwise warpgroups take them.
  if (warp < C::WARP_DQ) {
   reg_dealloc<C::REG_OTHER>();
   if (warp == C::WARP_TMA) {
    // ---------------------------------------------------------------- producer
    bool ok = true;
    int t = 0, u = 0, kv_issued = 0;
    const uint64_t stream_pol = policy_evict_first();  // inputs are read once: keep L2 for the dBias partials
    if (lane == 0) {
      tma_prefetch_map(&mQ);
      tma_prefetch_map(&mK);
      tma_prefetch_map(&mV);
      tma_prefetch_map(&mDO);
      tma_prefetch_map(&mBT);
    }
    for (int bi = 0; bi < nblk && ok; ++bi) {
      int hd, i0, nb;
      bool first;
      sc.block(bi, hd, i0, nb, first);
      const int b = hd / g.H, h = hd % g.H;
      for (int jt = 0; jt < njt && ok; ++jt) {
        for (int il = 0; il < nb; ++il, ++t) {
          const int st = t % C::NQS, i = i0 + il;
          if (t >= C::NQS) ok = wait_bar_warp(bar(C::B_QDOFREE + st), ((t / C::NQS) - 1) & 1, ab);
          if (!ok) break;
          {
            float *sl = reinterpret_cast<float *>(sm + C::OFF_LSE + st * 512);
            float *sd = reinterpret_cast<float *>(sm + C::OFF_D + st * 512);
            float lv[4], dvv[4];
            const int64_t lrow = (((int64_t)b * g.S + i) * g.H + h) * g.N;
#pragma unroll
            for (int m = 0; m < 4; ++m) {  // all loads first: one memory round trip
              const int j = jt * 128 + lane + 32 * m;
              lv[m] = j < g.N ? LSE[lrow + j] : -INFINITY;
              dvv[m] = j < g.N ? Dv[lrow + j] : 0.f;
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              sl[lane + 32 * m] = (lv[m] == -INFINITY) ? -INFINITY : -lv[m] * kLog2e;
              sd[lane + 32 * m] = dvv[m];
            }
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_QDOFULL + st), 2 * C::TILE);
            load_rows_hint(sb0 + C::OFF_Q + st * C::TILE, &mQ, bar(C::B_QDOFULL + st), NODE, h, b, g.S, i, jt * 128,
                           stream_pol);
            load_rows_hint(sb0 + C::OFF_DO + st * C::TILE, &mDO, bar(C::B_QDOFULL + st), NODE, h, b, g.S, i, jt * 128,
                           stream_pol);
          }
          if (jt == 0 && il == 0) {
            // K_i, V_i of the block (single-buffered: the previous block's MMAs must be done)
            if (bi > 0) ok = wait_bar_warp(bar(C::B_KVFREE), (bi - 1) & 1, ab);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * nb * C::TILE);
              for (int q = 0; q < nb; ++q) {
                load_rows_hint(sb0 + C::OFF_K + q * C::TILE, &mK, bar(C::B_KVFULL), NODE, h, b, g.S, i0 + q, kt * 128,
                               stream_pol);
                load_rows_hint(sb0 + C::OFF_V + q * C::TILE, &mV, bar(C::B_KVFULL), NODE, h, b, g.S, i0 + q, kt * 128,
                               stream_pol);
              }
            }
            kv_issued = bi + 1;
          }
          if (t == 0) {  // the first group's bias tile (the MMA warp loads the later ones)
            if (lane == 0) {
              const uint32_t dst = sb0 + C::OFF_BIAS;
              mbar_arrive_expect_tx(bar(C::B_BFULL), C::BIAS_TILE);
              tma_load_3d(dst, &mBT, bar(C::B_BFULL), jt * 128, kt * 128, b * g.H + h);
              tma_load_3d(dst + 16384, &mBT, bar(C::B_BFULL), jt * 128 + 64, kt * 128, b * g.H + h);
            }
            u = 1;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // drain copies still in flight before shared memory goes away
      if (kv_issued > 0) drain_bar(bar(C::B_KVFULL), (kv_issued - 1) & 1);
      if (u > 0) drain_bar(bar(C::B_BFULL), 0);
      for (int x = max(0, t - C::NQS); x < t; ++x) drain_bar(bar(C::B_QDOFULL + x % C::NQS), (x / C::NQS) & 1);
    }
   } else if (warp >= C::WARP_CV) {
    // ---------------------------------------------------------------- BF16 -> FP16 converters (+ mask rows)
    const int ct = tid - C::WARP_CV * 32;
    bool ok = true;
    int t = 0;
    for (int bi = 0; bi < nblk && ok; ++bi) {
      int hd, i0, nb;
      bool first;
      sc.block(bi, hd, i0, nb, first);
      const int b = hd / g.H;
      const BwdScales sc4 = load_scales<HD>(emax, hd);
      const float fk = exp2i(sc4.sk), fv = exp2i(sc4.sv), fq = exp2i(sc4.sq), fo = exp2i(sc4.so);
      ok = wait_bar_warp(bar(C::B_KVFULL), bi & 1, ab);
      if (!ok) break;
      // this warp's share of the block's K and V (the elementwise warps, idle at a block boundary,
      // convert the rest)
      convert_to_f16(sm + C::OFF_K, nb * C::TILE, fk, C::NEWT + ct, C::NEWT + C::NCVT);
      convert_to_f16(sm + C::OFF_V, nb * C::TILE, fv, C::NEWT + ct, C::NEWT + C::NCVT);
      float *maskf = reinterpret_cast<float *>(sm + C::OFF_MASK);
      for (int x = ct; x < nb * 128; x += C::NCVT) {
        const int il = x >> 7, k = kt * 128 + (x & 127);
        float mv = -INFINITY;  // keys past N are dead rows
        if (k < g.N) mv = mask ? bf16_to_f32(mask[((int64_t)b * g.S + i0 + il) * g.N + k]) * kLog2e : 0.f;
        maskf[x] = mv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_KVREADY));
      for (int jt = 0; jt < njt && ok; ++jt)
        for (int il = 0; il < nb; ++il, ++t) {
          const int st = t % C::NQS;
          ok = wait_bar_warp(bar(C::B_QDOFULL + st), (t / C::NQS) & 1, ab);
          if (!ok) break;
          convert_to_f16(sm + C::OFF_Q + st * C::TILE, C::TILE, fq, ct, C::NCVT);
          convert_to_f16(sm + C::OFF_DO + st * C::TILE, C::TILE, fo, ct, C::NCVT);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_QDOREADY + st));
        }
    }
   } else {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp walks the schedule converged (every decision is warp-uniform) and
    // elect.sync picks the lane that issues each MMA and commit.
    {
      constexpr uint32_t idSS = idesc_f16(128, 128, false, false, false, false);
      constexpr uint32_t idKV = idesc_f16(128, HD, false, false, false, true);
      constexpr uint32_t idQ = idesc_f16(128, HD, false, false, true, true);
      // descriptor bases: the start-address field is (address >> 4) in the low bits, so an operand
      // at base + off has descriptor base_desc + (off >> 4) (addresses stay below 256 KB)
      const uint64_t dK0 = smem_desc(sb0 + C::OFF_K, 16, 8 * C::ROWB, C::SW);
      const uint64_t dV0 = smem_desc(sb0 + C::OFF_V, 16, 8 * C::ROWB, C::SW);
      const uint64_t dQ0 = smem_desc(sb0 + C::OFF_Q, 16, 8 * C::ROWB, C::SW);
      const uint64_t dO0 = smem_desc(sb0 + C::OFF_DO, 16, 8 * C::ROWB, C::SW);
      const uint64_t dS0 = smem_desc(sb0 + C::OFF_DS, 1024, 2048, kSwizzle128B);
      constexpr uint64_t KS_ROW = (16 * C::ROWB) >> 4;  // 16 rows of an operand tile, descriptor units
      // per-step bookkeeping, walked in the common schedule
      int bi = 0, jt = 0, il = 0, hd = 0, nb = 0;
      {
        int i0;
        bool first;
        sc.block(0, hd, i0, nb, first);
      }
      auto advance = [&]() {
        if (++il == nb) {
          il = 0;
          if (++jt == njt) {
            jt = 0;
            ++bi;
            int i0;
            bool first;
            sc.block(bi, hd, i0, nb, first);
          }
        }
      };
      auto issue_s = [&](int il_, int st) {  // S^T = K_i Q_i^T
        const uint64_t a = dK0 + (uint64_t)((il_ * C::TILE) >> 4), b = dQ0 + (uint64_t)((st * C::TILE) >> 4);
        mma_ss_e(tb + C::TA, a, b, idSS, 0u);
#pragma unroll
        for (int ks = 1; ks < HD / 16; ++ks) mma_ss_e(tb + C::TA, a + 2 * ks, b + 2 * ks, idSS, 1u);
        mma_commit_e(bar(C::B_SFULL));
      };
      auto issue_dp = [&](int il_, int st) {  // dP^T = V_i dO_i^T
        const uint64_t a = dV0 + (uint64_t)((il_ * C::TILE) >> 4), b = dO0 + (uint64_t)((st * C::TILE) >> 4);
        mma_ss_e(tb + C::TB, a, b, idSS, 0u);
#pragma unroll
        for (int ks = 1; ks < HD / 16; ++ks) mma_ss_e(tb + C::TB, a + 2 * ks, b + 2 * ks, idSS, 1u);
        mma_commit_e(bar(C::B_DPFULL));
      };
      int ug = 0;  // query-tile groups finished: group ug's bias tile is in the buffer
      bool ok = wait_bar_warp(bar(C::B_KVREADY), 0, ab);
      if (ok) ok = wait_bar_warp(bar(C::B_QDOREADY), 0, ab);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_dp(0, 0);
      }
      for (int t = 0; t < T && ok; ++t) {
        const int st = t % C::NQS;
        const int cbi = bi, cjt = jt, cil = il;  // this step
        advance();                               // (bi, jt, il) now describe step t + 1
        const bool has_next = t + 1 < T;
        const bool next_new_block = has_next && jt == 0 && il == 0;
        const int st1 = (t + 1) % C::NQS;
        const uint32_t dcol = tb + C::TDKV + cil * 2 * HD;
        // ---- dV += P^T dO as soon as P^T is in region A (A operand: packed FP16 in TMEM)
        ok = wait_bar_warp(bar(C::B_PAFULL), t & 1, ab);
        if (ok && cjt == 0 && cil == 0 && cbi > 0) ok = wait_bar_warp(bar(C::B_DKVREAD), (cbi - 1) & 1, ab);
        if (ok && has_next && il == 0) {
          // the group's last P phase is done: every elementwise thread has released the bias tile
          // (before PAFULL), so the next group's tile (query tile jt of step t + 1) can be loaded
          ok = wait_bar_warp(bar(C::B_BFREE), ug & 1, ab);
          if (ok && lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_BFULL), C::BIAS_TILE);
            tma_load_3d(sb0 + C::OFF_BIAS, &mBT, bar(C::B_BFULL), jt * 128, kt * 128, hd);
            tma_load_3d(sb0 + C::OFF_BIAS + 16384, &mBT, bar(C::B_BFULL), jt * 128 + 64, kt * 128, hd);
          }
          __syncwarp();
          ++ug;
        }
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t b = dO0 + (uint64_t)((st * C::TILE) >> 4);
          // 16 queries per step: column group ks / KPG, packed columns (ks % KPG) * 8
          static_assert(C::KPG == 4 && C::QPT == 64, "P^T column pattern");
          mma_ts_x8_e<0, 8, 16, 24, 64, 72, 80, 88>(dcol + HD, tb + C::TA, b, KS_ROW, idKV, cjt > 0 ? 1u : 0u);
          mma_commit_e(bar(C::B_AFREE));
        }
        // ---- S^T(t+1) into region A right behind dV(t), which reads P^T from it: tcgen05.mma
        // operations issued by one thread are performed in issue order, so the write cannot overtake
        // the read and no completion wait is needed (within a block; a new block needs the new K, V)
        if (has_next && !next_new_block) {
          ok = wait_bar_warp(bar(C::B_QDOREADY + st1), ((t + 1) / C::NQS) & 1, ab);
          if (!ok) break;
          tc_fence_after();
          issue_s(il, st1);
        }
        // ---- dK += dS^T Q (A: packed FP16 dS^T in region B) and the dQ partial dS K (A: dS tile, MN-major)
        ok = wait_bar_warp(bar(C::B_PFULL), t & 1, ab);
        if (ok && t > 0) ok = wait_bar_warp(bar(C::B_DQREAD), (t - 1) & 1, ab);
        if (!ok) break;
        tc_fence_after();
        {
          const uint64_t bq = dQ0 + (uint64_t)((st * C::TILE) >> 4), bk = dK0 + (uint64_t)((cil * C::TILE) >> 4);
          mma_ts_x8_e<0, 8, 16, 24, 64, 72, 80, 88>(dcol, tb + C::TB, bq, KS_ROW, idKV, cjt > 0 ? 1u : 0u);
          mma_ss_x8_e(tb + C::TDQ, dS0, 4096 >> 4, bk, KS_ROW, idQ, 0u);
          mma_commit_e(bar(C::B_M2DONE));
          mma_commit_e(bar(C::B_QDOFREE + st));
          if (next_new_block || !has_next) mma_commit_e(bar(C::B_KVFREE));
        }
        if (has_next) {
          if (next_new_block) {
            ok = wait_bar_warp(bar(C::B_KVREADY), bi & 1, ab);
            if (ok) ok = wait_bar_warp(bar(C::B_QDOREADY + st1), ((t + 1) / C::NQS) & 1, ab);
            if (ok) ok = wait_bar_warp(bar(C::B_AFREE), t & 1, ab);
            if (!ok) break;
            tc_fence_after();
            issue_s(il, st1);
          }
          // ---- dP^T(t+1) once the dQ warps have read dQ(t) out of region B (tcgen05.ld by other
          // warps); dK(t), which reads dS^T from it, was issued earlier by this thread and is
          // performed first
          ok = wait_bar_warp(bar(C::B_DQREAD), t & 1, ab);
          if (!ok) break;
          tc_fence_after();
          issue_dp(il, st1);
        }
      }
      mma_commit_e(bar(C::B_FINAL));
      if (lane == 0) {
        drain_bar(bar(C::B_FINAL), 0);
        if (!ok && ug > 0) drain_bar(bar(C::B_BFULL), ug & 1);  // a bias load that no one waited for
      }
      __syncwarp();
    }
   }
  } else if (warp < C::WARP_EW0) {
    reg_dealloc<C::REG_DQ>();
    // ---------------------------------------------------------------- dQ warps: TMEM -> owners -> BF16
    const int dt = tid - C::WARP_DQ * 32;   // 0..127
    const int jl = (warp - C::WARP_DQ) * 32 + lane;  // query row of the partial = TMEM lane
    const uint32_t lb = (uint32_t)((warp - C::WARP_DQ) * 32) << 16;
    const uint32_t rb_bytes = (uint32_t)(nkt * (r1 - r0) * HD * 4);
    int o = (jl * nkt) >> 7;  // owner of row jl: o*128/n <= jl < (o+1)*128/n
    while (o + 1 < nkt && (int)((o + 1) * 128 / nkt) <= jl) ++o;
    while ((int)(o * 128 / nkt) > jl) --o;
    // step t's partial goes to receive slot t % NRB of its owner
    const uint32_t dst0 = mapa_shared(sb0 + C::OFF_RB + ((rank * rows_max + (jl - (int)(o * 128 / nkt))) * HD) * 4, o);
    const uint32_t rbar0 = mapa_shared(bar(C::B_RFULL), o);
    if (dt == 0)  // arm every slot for its first step
      for (int s = 0; s < C::NRB && s < T; ++s) mbar_arrive_expect_tx(bar(C::B_RFULL + s), rb_bytes);
    int prev_i = 0, prev_jt = 0, prev_hd = 0, red = 0;
    // the dQ factors of the blocks of slices (softmax scale / w, then 2^-sk), in this warp's two
    // shared-memory slots used by alternate blocks: the owner applies those of the step it sums
    float2 *dqf = reinterpret_cast<float2 *>(sm + C::OFF_DQF) + (warp - C::WARP_DQ) * 2;
    int pslot = 0;  // slot of the previous step's block
    auto reduce_prev = [&]() -> bool {
      const int slot = red % C::NRB;
      const float2 pf = dqf[pslot];
      if (!wait_bar_cluster_warp(bar(C::B_RFULL + slot), (red / C::NRB) & 1, ab)) return false;
      if (dt == 0 && red + C::NRB < T) mbar_arrive_expect_tx(bar(C::B_RFULL + slot), rb_bytes);  // arm its next step
      constexpr int CPR = HD / 4;
      const int items = (r1 - r0) * CPR;
      const float *rb = reinterpret_cast<const float *>(sm + C::OFF_RB + slot * C::RB_SLOT);
      for (int it = dt; it < items; it += C::NDQT) {
        const int rl = it / CPR, c = it % CPR;
        float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < nkt; ++r) {  // fixed order: key tile 0, 1, ..., n-1
          const float4 v = *reinterpret_cast<const float4 *>(rb + ((r * rows_max + rl) * HD + c * 4));
          s4.x += v.x;
          s4.y += v.y;
          s4.z += v.z;
          s4.w += v.w;
        }
        const int j = prev_jt * 128 + r0 + rl;
        if (j < g.N) {
          const uint2 w = make_uint2(
              pack_bf16x2(s4.x * pf.x * pf.y, s4.y * pf.x * pf.y), pack_bf16x2(s4.z * pf.x * pf.y, s4.w * pf.x * pf.y));
          *reinterpret_cast<uint2 *>(dQ + pos_row(g, prev_hd / g.H, prev_i, j, NODE) * g.H * HD + (prev_hd % g.H) * HD +
                                     c * 4) = w;
        }
      }
      __syncwarp();
      if (lane == 0)
        for (int r = 0; r < nkt; ++r) mbar_arrive_cluster_relaxed(mapa_shared(bar(C::B_XEMPTY + slot), r));
      ++red;
      return true;
    };
    bool ok = true;
    int t = 0;
    for (int bi = 0; bi < nblk && ok; ++bi) {
      int hd, i0, nb;
      bool first;
      sc.block(bi, hd, i0, nb, first);
      // the block's partials carry w 2^sk (all CTAs of the cluster work on the same head)
      if (lane == 0) {
        const BwdScales sc4 = load_scales<HD>(emax, hd);
        dqf[bi & 1] = make_float2(g.scale * exp2i(-(sc4.sv + sc4.so)), exp2i(-sc4.sk));
      }
      __syncwarp();
      for (int jt = 0; jt < njt && ok; ++jt)
        for (int il = 0; il < nb; ++il, ++t) {
          if (t > 0) {
            ok = reduce_prev();  // owner duty for the previous step (usually while this step's MMAs run)
            if (!ok) break;
          }
          ok = wait_bar_warp(bar(C::B_M2DONE), t & 1, ab);
          if (!ok) break;
          tc_fence_after();
          uint32_t r[HD];
          if constexpr (HD == 32) {
            tmem_ld32(tb + lb + C::TDQ, r);
          } else {
            tmem_ld16(tb + lb + C::TDQ, r);
          }
          tmem_wait_ld(r);
          tc_fence_before();
          mbar_arrive(bar(C::B_DQREAD));
          // slot t % NRB is free once every owner reduced step t - NRB from it
          if (t >= C::NRB) ok = wait_bar_cluster_warp(bar(C::B_XEMPTY + t % C::NRB), ((t / C::NRB) - 1) & 1, ab);
          if (!ok) break;
          {
            const uint32_t dst = dst0 + (t % C::NRB) * C::RB_SLOT, rbar = rbar0 + (t % C::NRB) * 8;
#pragma unroll
            for (int c = 0; c < HD / 4; ++c)
              st_async_f4(dst + c * 16, __uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]),
                          __uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3]), rbar);
          }
          prev_i = i0 + il;
          prev_jt = jt;
          prev_hd = hd;
          pslot = bi & 1;
        }
    }
    if (ok && red < T) ok = reduce_prev();  // the last step's rows
  } else {
    reg_alloc<C::REG_EW>();
    // ---------------------------------------------------------------- elementwise warps 8-15
    constexpr int QPT = C::QPT;
    const int ew = tid - C::WARP_EW0 * 32, ewarp = warp - C::WARP_EW0;  // 0..NEWT-1, 0..NEW-1
    const int q = warp & 3, cg = ewarp >> 2;  // TMEM lane quarter, column group of QPT queries
    const int hf = (cg * QPT) >> 6, c0 = ((cg * QPT) & 63) >> 3;  // query half, first 8-query chunk in it
    const int kl = q * 32 + lane;            // key row of the tile = TMEM lane
    const int kg = kt * 128 + kl;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const uint32_t colA = tb + lb + C::TA + cg * QPT, colB = tb + lb + C::TB + cg * QPT;
    const float c1 = g.scale * kLog2e;
    const float2 l2e2 = make_float2(kLog2e, kLog2e);
    const float *maskf = reinterpret_cast<const float *>(sm + C::OFF_MASK);
    // 8 queries per 16 bytes in the 128-byte-swizzled tiles: row of key kl, chunk c at ((c ^ (kl & 7)) << 4)
    const uint32_t trow = (kl >> 3) * 2048 + hf * 1024 + (kl & 7) * 128;
    bool ok = true;
    int t = 0, u = 0;
    float2 acc[QPT / 2];  // dBias tile row: queries cg*QPT + [0,QPT) as pairs
    for (int bi = 0; bi < nblk && ok; ++bi) {
      int hd, i0, nb;
      bool first;  // the block opens its head's segment: the partial tiles start from zero
      sc.block(bi, hd, i0, nb, first);
      const int b = hd / g.H, h = hd % g.H;
      // the head's operand scales: S^T carries 2^(sk+sq), dP^T and the dBias sums carry w = 2^(sv+so)
      float2 c12, mw2;
      {
        const BwdScales sc4 = load_scales<HD>(emax, hd);
        const float c1s = c1 * exp2i(-(sc4.sk + sc4.sq)), wv = exp2i(sc4.sv + sc4.so);
        c12 = make_float2(c1s, c1s);
        mw2 = make_float2(-wv, -wv);
      }
      // this cluster's dBias partial slot for head hd: slot k = cl - (first cluster of the head),
      // tiles [head][slot][kt][jt][128 x 128]
      const int64_t pslot = ((int64_t)hd * KMAX + (cl - bwd_cluster_of((int64_t)hd * g.S, NC, W))) * nkt * njt;
      auto ptile = [&](int jt_) -> int64_t { return (pslot + (int64_t)kt * njt + jt_) * 16384; };
      // help convert the block's K and V to FP16 (with the converter warps), then wait until the whole
      // conversion and the block's mask rows are in place
      ok = wait_bar_warp(bar(C::B_KVFULL), bi & 1, ab);
      if (!ok) break;
      {
        const BwdScales sc4 = load_scales<HD>(emax, hd);
        convert_to_f16(sm + C::OFF_K, nb * C::TILE, exp2i(sc4.sk), ew, C::NEWT + C::NCVT);
        convert_to_f16(sm + C::OFF_V, nb * C::TILE, exp2i(sc4.sv), ew, C::NEWT + C::NCVT);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_KVREADY));
      ok = wait_bar_warp(bar(C::B_KVREADY), bi & 1, ab);
      for (int jt = 0; jt < njt && ok; ++jt) {
        ok = wait_bar_warp(bar(C::B_BFULL), u & 1, ab);
        if (!ok) break;
#pragma unroll
        for (int e = 0; e < QPT / 2; ++e) acc[e] = make_float2(0.f, 0.f);
        const uint32_t brow = sb0 + C::OFF_BIAS + hf * 16384 + kl * 128;
        for (int il = 0; il < nb; ++il, ++t) {
          const int st = t % C::NQS;
          // mask*log2e of this key (-inf for masked keys and keys past N: their exponent is -inf, P = +0)
          const float mk = maskf[il * 128 + kl];
          const bool unmasked = __all_sync(0xffffffffu, mk == 0.f);  // warp-uniform: skip the mask add
          const float2 mk2 = make_float2(mk, mk);
          const float *sl = reinterpret_cast<const float *>(sm + C::OFF_LSE + st * 512) + cg * QPT;
          const float *sd = reinterpret_cast<const float *>(sm + C::OFF_D + st * 512) + cg * QPT;
          if (il == nb - 1 && !first)  // the warp's QPT/8 KB of the dBias partial tile into L2 ahead of the flush
#pragma unroll
            for (int r = 0; r < QPT / 32; ++r) {
              const int li = lane + 32 * r;  // 128-byte line li of the warp's chunks
              prefetch_l2_keep(partial + ptile(jt) + ((hf * 8 + c0 + (li >> 3)) * 128 + q * 32) * 8 + (li & 7) * 32);
            }
          ok = wait_bar_warp(bar(C::B_SFULL), t & 1, ab);
          if (!ok) break;
          tc_fence_after();
          uint32_t pw[QPT / 2];  // P as FP16 pairs: the P^T operand and the factor of dS
#pragma unroll
          for (int hh = 0; hh < QPT / 32; ++hh) {  // 32 queries at a time
            uint32_t pv[32];                       // S^T values
            tmem_ld32(colA + hh * 32, pv);
            tmem_wait_ld(pv);
#pragma unroll
            for (int mq = 0; mq < 4; ++mq) {  // 8 queries (one 16-byte bias chunk) at a time
              const int m = hh * 4 + mq;
              uint32_t bw[4];
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(bw[0]), "=r"(bw[1]), "=r"(bw[2]), "=r"(bw[3])
                           : "r"(brow + (((c0 + m) ^ (kl & 7)) << 4)));
              const float4 u0 = reinterpret_cast<const float4 *>(sl)[2 * m];
              const float4 u1 = reinterpret_cast<const float4 *>(sl)[2 * m + 1];
              const float2 uu[4] = {make_float2(u0.x, u0.y), make_float2(u0.z, u0.w), make_float2(u1.x, u1.y),
                                    make_float2(u1.z, u1.w)};
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const int x = mq * 8 + 2 * e2;
                const float2 bv = make_float2(__uint_as_float(bw[e2] << 16), __uint_as_float(bw[e2] & 0xffff0000u));
                const float2 base = __ffma2_rn(bv, l2e2, unmasked ? uu[e2] : __fadd2_rn(uu[e2], mk2));
                const float2 arg = __ffma2_rn(make_float2(__uint_as_float(pv[x]), __uint_as_float(pv[x + 1])), c12, base);
                pw[m * 4 + e2] = pack_f16x2(ex2(arg.x), ex2(arg.y));
              }
            }
          }
          if (il == nb - 1) {  // this group's bias tile is no longer read: hand it back to the TMA
            fence_proxy_async_smem();  // order these generic-proxy reads before the async-proxy overwrite
            mbar_arrive(bar(C::B_BFREE));
          }
          if constexpr (QPT == 64) {  // P^T (FP16 pairs) over this thread's S^T columns: the A operand of dV
            tmem_st32(colA, pw);
          } else {
            tmem_st16(colA, pw);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::B_PAFULL));
          ok = wait_bar_warp(bar(C::B_DPFULL), t & 1, ab);  // (also: dQ of the previous step has read the dS tile)
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c2 = 0; c2 < QPT / 16; ++c2) {  // 16 queries at a time
            uint32_t dv[16];
            tmem_ld16(colB + c2 * 16, dv);
            tmem_wait_ld(dv);
            uint32_t dw[8];  // dS as FP16 pairs
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2) {
              const int x0 = c2 * 16 + 2 * e2;
              const float2 dd = reinterpret_cast<const float2 *>(sd)[x0 >> 1];
              const float2 dp = make_float2(__uint_as_float(dv[2 * e2]), __uint_as_float(dv[2 * e2 + 1]));
              const float2 pp = __half22float2(*reinterpret_cast<const __half2 *>(&pw[x0 >> 1]));
              const float2 ds = __fmul2_rn(pp, __ffma2_rn(dd, mw2, dp));  // p (dp - w D) = w dS
              acc[x0 >> 1] = __fadd2_rn(acc[x0 >> 1], ds);
              dw[e2] = pack_f16x2(ds.x, ds.y);
            }
            tmem_st8(colB + c2 * 8, dw);  // dS^T (FP16 pairs) over columns already read: the A operand of dK
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {  // and into the dS tile, the A operand of dQ
              const int m = c2 * 2 + cc;
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sb0 + C::OFF_DS + trow + (((c0 + m) ^ (kl & 7)) << 4)),
                           "r"(dw[4 * cc]), "r"(dw[4 * cc + 1]), "r"(dw[4 * cc + 2]), "r"(dw[4 * cc + 3])
                           : "memory");
            }
          }
          fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::B_PFULL));
        }
        if (!ok) break;
        // ---- dBias tile (jt, kt) of this block into the cluster's partial slot (FP32, owned by this CTA).
        // Tile layout [query half][chunk c of 8 queries][key][8 queries]: lane-consecutive keys make
        // every warp access one contiguous kilobyte.
        if (kg < g.N) {
          float *pp = partial + ptile(jt) + ((hf * 8 + c0) * 128 + kl) * 8;  // chunk c0 + m at + m * 1024
          uint32_t w[QPT / 8][8];  // all the 32-byte loads in flight at once, then add and store
#pragma unroll
          for (int m = 0; m < QPT / 8; ++m) {
            if (!first) {
              ld_keep_v8(pp + 1024 * m, w[m]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) w[m][e] = 0u;
            }
          }
          const float iw = __frcp_rn(-mw2.x);  // the register sums carry w (a power of two: exact)
#pragma unroll
          for (int m = 0; m < QPT / 8; ++m) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 a = acc[4 * m + e];
              w[m][2 * e] = __float_as_uint(fmaf(a.x, iw, __uint_as_float(w[m][2 * e])));
              w[m][2 * e + 1] = __float_as_uint(fmaf(a.y, iw, __uint_as_float(w[m][2 * e + 1])));
            }
            st_keep_v8(pp + 1024 * m, w[m]);
          }
        }
        ++u;
      }
      if (!ok) break;
      // ---- dK_i, dV_i of the block -> BF16, once the block's last MMAs are complete: column group 0
      // writes dK, group 1 dV. Each warp stages its 32 key rows of a slice in its own 2 KB piece of
      // the dS tile (free now; two pieces per warp, used alternately over the slices), in the TMA
      // swizzle, and stores them with one 32-row TMA box; rows past N are clipped by the TMA.
      ok = wait_bar_warp(bar(C::B_M2DONE), (t - 1) & 1, ab);
      if (!ok) break;
      tc_fence_after();
      {
        static_assert(C::NEW == 8 && 2 * C::NEW * 32 * C::ROWB <= 32768, "dK/dV staging in the dS tile");
        const CUtensorMap *mo = cg == 0 ? &mDK : &mDV;
        // 16-byte chunk c of staged row lane: SW64 (64-byte rows) or SW32 (32-byte rows)
        const uint32_t swz = HD == 32 ? (uint32_t)((lane >> 1) & 3) : (uint32_t)((lane >> 2) & 1);
        for (int il = 0; il < nb; ++il) {
          // dK carries w 2^sq (and takes the softmax scale), dV carries 2^so
          const BwdScales sc4 = load_scales<HD>(emax, hd);
          const float f = cg == 0 ? g.scale * exp2i(-(sc4.sv + sc4.so)) : exp2i(-sc4.so);
          const float f2 = cg == 0 ? exp2i(-sc4.sq) : 1.f;  // (dK: the third factor, applied separately)
          uint32_t r[HD];
          const uint32_t col = tb + lb + C::TDKV + il * 2 * HD + cg * HD;
          if constexpr (HD == 32) {
            tmem_ld32(col, r);
          } else {
            tmem_ld16(col, r);
          }
          tmem_wait_ld(r);
          uint32_t w[HD / 2];
#pragma unroll
          for (int c = 0; c < HD / 2; ++c)
            w[c] = pack_bf16x2(__uint_as_float(r[2 * c]) * f * f2, __uint_as_float(r[2 * c + 1]) * f * f2);
          if (il >= 2) {  // the store of slice il - 2 has read this piece
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
          }
          const uint32_t piece = sb0 + C::OFF_DS + (ewarp * 2 + (il & 1)) * (32 * C::ROWB);
#pragma unroll
          for (int c = 0; c < HD / 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(piece + lane * C::ROWB + ((c ^ swz) << 4)),
                         "r"(w[4 * c]), "r"(w[4 * c + 1]), "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                         : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            store_rows(mo, piece, NODE, h, b, g.S, i0 + il, kt * 128 + q * 32);
            bulk_commit_group();
          }
        }
        if (lane == 0) bulk_wait_group_read<0>();  // the next block's dS tiles overwrite these pieces
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DKVREAD));
    }
  }
  if (warp >= C::WARP_EW0 && lane == 0) bulk_wait_group<0>();  // the dK, dV stores have been performed
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still write or read its shared memory
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tb, C::TMEM_COLS);
  }
}

// biasT[bh][k][j] = bias[bh][j][k] for j, k < N, zero in the padding up to NP; also zeroes the
// head's four exponent maxima that the preparation kernel accumulates next.
__global__ void bias_transpose_kernel(const uint16_t *__restrict__ bias, uint16_t *__restrict__ biasT, int N,
                                      int NP, int *__restrict__ emax) {
  __shared__ uint16_t tile[32][33];
  const int bh = blockIdx.z, j0 = blockIdx.y * 32, k0 = blockIdx.x * 32;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.y == 0 && threadIdx.x < 4) emax[4 * bh + threadIdx.x] = 0;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int j = j0 + r, k = k0 + threadIdx.x;
    tile[r][threadIdx.x] = (j < N && k < N) ? bias[((int64_t)bh * N + j) * N + k] : (uint16_t)0;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int k = k0 + r, j = j0 + threadIdx.x;
    biasT[((int64_t)bh * NP + k) * NP + j] = tile[threadIdx.x][r];
  }
}

// dBias[bh][j][k] = BF16(sum, in cluster order, of the partials of head bh): the clusters whose
// ranges hold slices of head bh wrote slots 0, 1, ... of the head. Each slot holds tiles [kt][jt] of
// 128 keys x 128 queries laid out [query half][chunk c][key][8 queries].
// One CTA (256 threads) reduces one [128 keys x 8 queries] chunk and writes its 8 output rows.
__global__ void dbias_reduce_t_kernel(const float *__restrict__ partial, int NC, int KMAX, int S, int64_t W, int N,
                                      int NP, uint16_t *__restrict__ dBias) {
  __shared__ float s[8][129];
  const int nt = NP / 128, tile = blockIdx.x, kt = tile / nt, jt = tile % nt;
  const int hc = blockIdx.y, bh = blockIdx.z, tid = threadIdx.x;
  const int nslots = bwd_cluster_of((int64_t)bh * S + S - 1, NC, W) - bwd_cluster_of((int64_t)bh * S, NC, W) + 1;
  const int64_t sstride4 = (int64_t)nt * nt * 16384 / 4;
  const int kl = tid >> 1, e0 = (tid & 1) * 4;
  if (kt * 128 + kl < N) {
    const float4 *p = reinterpret_cast<const float4 *>(partial + ((int64_t)bh * KMAX * nt * nt + tile) * 16384 +
                                                       (hc * 128 + kl) * 8 + e0);
    float4 a = __ldcs(p);
    for (int gi = 1; gi < nslots; ++gi) {
      const float4 v = __ldcs(p + gi * sstride4);
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    s[e0][kl] = a.x;
    s[e0 + 1][kl] = a.y;
    s[e0 + 2][kl] = a.z;
    s[e0 + 3][kl] = a.w;
  }
  __syncthreads();
  const int e = tid >> 5, j = jt * 128 + hc * 8 + e;
  if (j < N)
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int kk = (tid & 31) + 32 * m, k = kt * 128 + kk;
      if (k < N) dBias[((int64_t)bh * N + j) * N + k] = f32_to_bf16_rn(s[e][kk]);
    }
}

cudaError_t launch_bias_transpose(const Dims &g, const uint16_t *bias, uint16_t *biasT, int *emax,
                                  cudaStream_t stream) {
  const int NP = (g.N + 127) / 128 * 128;
  dim3 grid(NP / 32, NP / 32, g.B * g.H), block(32, 8);
  bias_transpose_kernel<<<grid, block, 0, stream>>>(bias, biasT, g.N, NP, emax);
  return cudaGetLastError();
}

cudaError_t launch_dbias_reduce_t(const Dims &g, const BwdSplit &sp, const float *partial, uint16_t *dBias,
                                  cudaStream_t stream) {
  const int NP = (g.N + 127) / 128 * 128;
  const int nt = NP / 128;
  dim3 grid(nt * nt, 16, g.B * g.H);
  dbias_reduce_t_kernel<<<grid, 256, 0, stream>>>(partial, sp.NC, sp.KMAX, g.S, (int64_t)g.B * g.H * g.S, g.N, NP,
                                                  dBias);
  return cudaGetLastError();
}

template <int HD>
cudaError_t plan_bwd_t(const Dims &g, const BwdSplit &sp, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                       const uint16_t *dO, const uint16_t *biasT, uint16_t *dK, uint16_t *dV, BwdPlan *p) {
  using C = BwdCfg<HD>;
  const int nkt = (g.N + 127) / 128, NP = nkt * 128;
  p->sp = sp;
  cudaError_t e = make_rows_map(&p->mq, Q, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&p->mdk, dK, g, 32);
  if (e == cudaSuccess) e = make_rows_map(&p->mdv, dV, g, 32);
  if (e == cudaSuccess) e = make_rows_map(&p->mk, K, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&p->mv, V, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&p->mdo, dO, g, 128);
  if (e == cudaSuccess) e = make_square_map(&p->mbt, biasT, NP, g.B * g.H);
  if (e != cudaSuccess) return e;
  auto *kern = g.node ? bwd_kernel<HD, 1> : bwd_kernel<HD, 0>;
  int dev = 0;
  e = current_device(&dev);
  if (e != cudaSuccess) return e;
  static DeviceOnce ready[2];  // per node
  DeviceOnce &once = ready[g.node ? 1 : 0];
  if (!once.done(dev)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    // The setmaxnreg split moves registers between warpgroups within the block's
    // launch allocation; it only balances if the kernel was built with exactly
    // REG_LAUNCH registers per thread, so refuse to launch otherwise.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != (int)C::REG_LAUNCH) return cudaErrorInvalidConfiguration;
    once.mark(dev);
  }
  return cudaSuccess;
}

cudaError_t plan_bwd(const Dims &g, const BwdSplit &sp, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     const uint16_t *dO, const uint16_t *biasT, uint16_t *dK, uint16_t *dV, BwdPlan *p) {
  return g.d == 32 ? plan_bwd_t<32>(g, sp, Q, K, V, dO, biasT, dK, dV, p)
                   : plan_bwd_t<16>(g, sp, Q, K, V, dO, biasT, dK, dV, p);
}

template <int HD>
static cudaError_t launch_bwd_main_t(const Dims &g, const BwdPlan &p, const float *LSE, const float *Dv,
                                     const int *emax, const uint16_t *mask, uint16_t *dQ, uint16_t *dK, uint16_t *dV,
                                     float *partial, int *status, cudaStream_t stream) {
  using C = BwdCfg<HD>;
  const int nkt = (g.N + 127) / 128;
  auto *kern = g.node ? bwd_kernel<HD, 1> : bwd_kernel<HD, 0>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nkt, p.sp.NC, 1);
  cfg.blockDim = dim3(C::NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = nkt;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p.mq, p.mk, p.mv, p.mdo, p.mbt, p.mdk, p.mdv, g, p.sp.NC, p.sp.KMAX, LSE, Dv,
                            emax, mask, dQ, dK, dV, partial, status);
}

cudaError_t launch_bwd_main(const Dims &g, const BwdPlan &p, const float *LSE, const float *Dv, const int *emax,
                            const uint16_t *mask, uint16_t *dQ, uint16_t *dK, uint16_t *dV, float *partial,
                            int *status, cudaStream_t stream) {
  if (g.d == 32) return launch_bwd_main_t<32>(g, p, LSE, Dv, emax, mask, dQ, dK, dV, partial, status, stream);
  return launch_bwd_main_t<16>(g, p, LSE, Dv, emax, mask, dQ, dK, dV, partial, status, stream);
}

// Streaming multiprocessors of the current device (cached per device).
cudaError_t device_sm_count(int *nsm) {
  static DeviceValue cache;
  int dev = 0;
  cudaError_t e = current_device(&dev);
  if (e != cudaSuccess) return e;
  int n = cache.get(dev);
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidDevice;
    cache.set(dev, n);
  }
  *nsm = n;
  return cudaSuccess;
}

// Most clusters a shape is split over on a device with nsm SMs: one per nkt SMs, never more than
// the number of (head, slice) pairs (so that every cluster has at least one slice).
int bwd_clusters_max(const Dims &g, int nsm) {
  const int nkt = (g.N + 127) / 128;
  const int64_t W = (int64_t)g.B * g.H * g.S;
  int n = nsm / nkt;
  if (n < 1) n = 1;
  return (int)(W < n ? W : n);
}

// dBias partial slots one head needs when the work is split over NC clusters: the most clusters
// whose ranges hold slices of one head. Only heads that contain a range boundary can reach more
// than one, so it suffices to look at those.
int bwd_slots_for(const Dims &g, int NC) {
  const int64_t W = (int64_t)g.B * g.H * g.S;
  int k = 1;
  for (int c = 1; c < NC; ++c) {
    const int64_t hd = bwd_unit_start(c, NC, W) / g.S;
    const int n = bwd_cluster_of(hd * g.S + g.S - 1, NC, W) - bwd_cluster_of(hd * g.S, NC, W) + 1;
    if (n > k) k = n;
  }
  return k;
}

// Slots per head the workspace holds: enough for any split over at most bwd_clusters_max clusters
// of a device with nsm SMs.
int bwd_slots_max(const Dims &g, int nsm) {
  int k = 1;
  for (int nc = 1; nc <= bwd_clusters_max(g, nsm); ++nc) {
    const int s = bwd_slots_for(g, nc);
    if (s > k) k = s;
  }
  return k;
}

// Clusters of nkt CTAs the device runs at once for this kernel (cached per device).
template <int HD>
cudaError_t bwd_resident_clusters_t(const Dims &g, int *out) {
  using C = BwdCfg<HD>;
  static DeviceValue cache[9];  // [cluster size][device]
  const int nkt = (g.N + 127) / 128;
  int dev = 0;
  cudaError_t e = current_device(&dev);
  if (e != cudaSuccess) return e;
  int n = cache[nkt].get(dev);
  if (n == 0) {
    // (both node instantiations have the same resources: the starting-node one stands for them)
    e = cudaFuncSetAttribute(bwd_kernel<HD, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nkt, 1, 1);
    cfg.blockDim = dim3(C::NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = nkt;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&n, bwd_kernel<HD, 0>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;  // not even one cluster fits on this device
    cache[nkt].set(dev, n);
  }
  *out = n;
  return cudaSuccess;
}

// The split a call uses: as many clusters as the device runs at once (one wave), within the
// workspace bound. Depends only on the shape and the device (its SM count and how many of the
// kernel's clusters it keeps resident), so repeated calls reduce in the same order. Fails, rather
// than falling back to another split, when the device cannot be queried.
cudaError_t bwd_split_active(const Dims &g, BwdSplit *sp) {
  int n = 0, nsm = 0;
  cudaError_t e = g.d == 32 ? bwd_resident_clusters_t<32>(g, &n) : bwd_resident_clusters_t<16>(g, &n);
  if (e == cudaSuccess) e = device_sm_count(&nsm);
  if (e != cudaSuccess) return e;
  const int cmax = bwd_clusters_max(g, nsm);
  sp->NC = n < cmax ? n : cmax;
  sp->KMAX = bwd_slots_for(g, sp->NC);
  return cudaSuccess;
}

}  // namespace triattn
