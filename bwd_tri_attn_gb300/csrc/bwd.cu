// Backward pass: key-tile-parallel tcgen05 kernel that recomputes every
// probability tile exactly once and produces dQ, dK, dV and the dBias partials.
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract): the shared pair bias adds a
// reduction over slices to the usual reductions over queries (dK, dV) and keys
// (dQ); the key-tile-parallel backward recomputes each probability tile once
// and uses ordered partial reductions, with no floating-point atomics and no
// full score-gradient storage.
//
// Work unit (one CTA): batch b, head h, key tile kt (128 keys), and a
// "supergroup" of consecutive slices, walked in blocks of GB slices:
//     for block: for query tile jt: for slice i in block:
//         S^T  = K_i Q_i[jt]^T        (TMEM, lanes = keys)
//         dP^T = V_i dO_i[jt]^T
//         P^T  = exp2(S^T*scale*log2e + biasT*log2e - LSE*log2e)   (FP32, written back as FP16)
//         dS^T = P^T * (dP^T - D)
//         dV_i += P^T dO_i[jt],  dK_i += dS^T Q_i[jt]            (TMEM accumulators, one pair per slice of the block)
//         dQ_i[jt] partial = dS K_i                               (reduced across the cluster, below)
//         dBias tile (jt, kt) += dS   (registers, summed in slice order over the block)
//     after each (block, jt): the dBias tile is added into the supergroup's FP32 partial (this CTA owns it)
//     after each block: dK_i, dV_i -> BF16
//
// Three reductions, each in a fixed order:
//  - dK, dV over query tiles: in the CTA's TMEM accumulator, jt = 0, 1, ...
//  - dQ over key tiles: the n = N/128 CTAs of one (b, h, supergroup) form a
//    thread-block cluster. CTA r owns query rows [r*128/n, (r+1)*128/n) of every
//    step's tile; each CTA pushes the matching rows of its 128 x d FP32 partial
//    into the owner's receive buffer with st.async (completing bytes on the
//    owner's mbarrier), and the owner sums the n partials in rank (= kt) order,
//    one step later so that the exchange overlaps the next step's work.
//  - dBias over slices: within a block in slice order (registers), across blocks in
//    block order (the partial), across supergroups in supergroup order (reduce kernel).
// Every order depends on the shape only.
//
// Operands: all tensor-core operands are FP16 (Q, K, V, dO converted in shared
// memory, exact in the FP16 range); P and dS need FP16's 11-bit significand.
//
// Warps: 0-7 elementwise (thread = key row x 64 query columns; warp w uses the
// TMEM lane quarter w % 4 and query half w / 4), 8 = TMA producer, 9 = MMA issuer.
// TMEM: [0,128) S^T, overwritten in place by P^T (FP16 pairs: queries 0-63 in
// cols 0-31, queries 64-127 in cols 64-95, so each query half writes only
// columns it has already read) and then by the dQ partial (cols 96..96+d);
// [128,256) dP^T then dS^T (same packing); 256 + 2*d*il: dK_il, dV_il.
#include "common.cuh"
#include "sm100.cuh"
#include "sync.cuh"
#include "tmap.cuh"

namespace triattn {
using namespace sm100;

template <int HD>
struct BwdCfg {
  static constexpr int GB = HD == 32 ? 4 : 8;  // slices per block: GB * 2d TMEM columns of dK/dV
  static constexpr int NQS = 2;                // Q/dO stages
  static constexpr int ROWB = HD * 2;
  static constexpr int TILE = 128 * ROWB;
  static constexpr uint32_t SW = HD == 32 ? kSwizzle64B : kSwizzle32B;
  static constexpr int NEW = 8;  // elementwise warps
  static constexpr int NEWT = NEW * 32;
  static constexpr int WARP_TMA = NEW, WARP_MMA = NEW + 1;
  static constexpr int NTHREADS = (NEW + 2) * 32;
  static constexpr int BIAS_TILE = 128 * 128 * 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + GB * TILE;
  static constexpr int OFF_Q = OFF_V + GB * TILE;
  static constexpr int OFF_DO = OFF_Q + NQS * TILE;
  static constexpr int OFF_BIAS = OFF_DO + NQS * TILE;     // 2 x [2 halves][128 rows][128 B], SW128
  static constexpr int OFF_DS = OFF_BIAS + 2 * BIAS_TILE;  // FP16 dS, MN-major SW128: [16 key groups][2][8][128 B]
  static constexpr int RB_ROWS = 136;                      // >= n * ceil(128 / n) for every cluster size n <= 8
  static constexpr int OFF_RB = OFF_DS + 32768;            // dQ receive buffer: [sender][row][HD] FP32
  static constexpr int OFF_LSE = OFF_RB + RB_ROWS * HD * 4; // [NQS][128]: -LSE*log2e (or -inf)
  static constexpr int OFF_D = OFF_LSE + NQS * 512;        // [NQS][128]: D
  static constexpr int OFF_MASK = OFF_D + NQS * 512;       // [GB][128]: mask*log2e of this CTA's keys
  static constexpr int OFF_BAR = OFF_MASK + GB * 512;
  static constexpr int B_KVFULL = 0, B_KVREADY = 1, B_KVFREE = 2;
  static constexpr int B_QDOFULL = 3, B_QDOREADY = B_QDOFULL + NQS, B_QDOFREE = B_QDOREADY + NQS;
  static constexpr int B_BFULL = B_QDOFREE + NQS, B_BFREE = B_BFULL + 2;
  static constexpr int B_SFULL = B_BFREE + 2, B_PFULL = B_SFULL + 1, B_M2DONE = B_PFULL + 1;
  static constexpr int B_DQREAD = B_M2DONE + 1, B_DKVREAD = B_DQREAD + 1;
  static constexpr int B_RFULL = B_DKVREAD + 1, B_XEMPTY = B_RFULL + 1, B_FINAL = B_XEMPTY + 1;
  static constexpr int NBAR = B_FINAL + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(256 + GB * 2 * HD <= 512, "TMEM budget");
  static_assert(OFF_BIAS % 1024 == 0 && OFF_DS % 1024 == 0, "SW128 tiles need 1 KB alignment");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Upper bound on the number of slice supergroups (dBias partials) for a shape:
// clusters of N/128 CTAs filling at most 152 SMs once, never more than the
// number of slice blocks. The workspace is sized for this bound.
inline int bwd_supergroups_max(const Dims &g) {
  const int nkt = (g.N + 127) / 128;
  const int gb = g.d == 32 ? BwdCfg<32>::GB : BwdCfg<16>::GB;
  const int blocks = (g.S + gb - 1) / gb;
  int gp = 152 / (nkt * g.B * g.H);
  if (gp < 1) gp = 1;
  if (gp > blocks) gp = blocks;
  return gp;
}

__device__ __forceinline__ bool wait_bar_cluster_warp(uint32_t bar, uint32_t parity, const Abort &ab) {
  const bool ok = wait_bar_cluster(bar, parity, ab);
  return __all_sync(0xffffffffu, ok);
}

// BF16 -> FP16 in place over `bytes` of shared memory, split across `nthr` threads.
__device__ __forceinline__ void convert_to_f16(uint8_t *p, int bytes, int tid, int nthr) {
  uint4 *v = reinterpret_cast<uint4 *>(p);
  for (int e = tid; e < bytes / 16; e += nthr) {
    uint4 w = v[e];
    w.x = bf16x2_to_f16x2(w.x);
    w.y = bf16x2_to_f16x2(w.y);
    w.z = bf16x2_to_f16x2(w.z);
    w.w = bf16x2_to_f16x2(w.w);
    v[e] = w;
  }
}

template <int HD>
__global__ void __launch_bounds__(BwdCfg<HD>::NTHREADS, 1)
bwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
           const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mDO,
           const __grid_constant__ CUtensorMap mBT, const Dims g, const int Gp, const float *__restrict__ LSE,
           const float *__restrict__ Dv, const uint16_t *__restrict__ mask, uint16_t *__restrict__ dQ,
           uint16_t *__restrict__ dK, uint16_t *__restrict__ dV, float *__restrict__ partial, int *status) {
  using C = BwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkt = (g.N + 127) / 128, njt = nkt, NP = nkt * 128;
  const int kt = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / Gp, grp = blockIdx.z % Gp;
  const uint32_t rank = cluster_ctarank();  // == kt (cluster spans the key tiles)
  const int s0 = (int)((int64_t)grp * g.S / Gp), s1 = (int)((int64_t)(grp + 1) * g.S / Gp);
  const int nblk = (s1 - s0 + C::GB - 1) / C::GB;
  const int T = njt * (s1 - s0);  // steps of this CTA
  auto bar = [&](int k) { return sb0 + C::OFF_BAR + 8u * (uint32_t)k; };
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_MISC);
  const Abort ab{reinterpret_cast<volatile int *>(misc + 1), status};

  if (tid == 0) {
    mbar_init(bar(C::B_KVFULL), 1);
    mbar_init(bar(C::B_KVREADY), C::NEWT);
    mbar_init(bar(C::B_KVFREE), 1);
    for (int s = 0; s < C::NQS; ++s) {
      mbar_init(bar(C::B_QDOFULL + s), 1);
      mbar_init(bar(C::B_QDOREADY + s), C::NEWT);
      mbar_init(bar(C::B_QDOFREE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_BFULL + s), 1);
      mbar_init(bar(C::B_BFREE + s), C::NEWT);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_PFULL), C::NEWT);
    mbar_init(bar(C::B_M2DONE), 1);
    mbar_init(bar(C::B_DQREAD), C::NEWT);
    mbar_init(bar(C::B_DKVREAD), C::NEWT);
    mbar_init(bar(C::B_RFULL), 1);             // + the bytes pushed by all n senders
    mbar_init(bar(C::B_XEMPTY), C::NEW * nkt);  // one arrive per elementwise warp of every owner
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

  if (warp == C::WARP_TMA) {
    // ---------------------------------------------------------------- producer
    bool ok = true;
    int t = 0, u = 0, kv_issued = 0;
    if (lane == 0) {
      tma_prefetch_map(&mQ);
      tma_prefetch_map(&mK);
      tma_prefetch_map(&mV);
      tma_prefetch_map(&mDO);
      tma_prefetch_map(&mBT);
    }
    for (int bi = 0; bi < nblk && ok; ++bi) {
      const int i0 = s0 + bi * C::GB, nb = min(C::GB, s1 - i0);
      for (int jt = 0; jt < njt && ok; ++jt) {
        for (int il = 0; il < nb; ++il, ++t) {
          const int st = t % C::NQS, i = i0 + il;
          if (t >= C::NQS) ok = wait_bar_warp(bar(C::B_QDOFREE + st), ((t / C::NQS) - 1) & 1, ab);
          if (!ok) break;
          float *sl = reinterpret_cast<float *>(sm + C::OFF_LSE + st * 512);
          float *sd = reinterpret_cast<float *>(sm + C::OFF_D + st * 512);
          {
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
            tma_load_4d(sb0 + C::OFF_Q + st * C::TILE, &mQ, bar(C::B_QDOFULL + st), 0, h, jt * 128, b * g.S + i);
            tma_load_4d(sb0 + C::OFF_DO + st * C::TILE, &mDO, bar(C::B_QDOFULL + st), 0, h, jt * 128, b * g.S + i);
          }
          if (jt == 0 && il == 0) {
            // K_i, V_i of the block (single-buffered: wait until the previous block's MMAs are done)
            if (bi > 0) ok = wait_bar_warp(bar(C::B_KVFREE), (bi - 1) & 1, ab);
            if (!ok) break;
            if (lane == 0) {
              mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * nb * C::TILE);
              for (int q = 0; q < nb; ++q) {
                tma_load_4d(sb0 + C::OFF_K + q * C::TILE, &mK, bar(C::B_KVFULL), 0, h, kt * 128, b * g.S + i0 + q);
                tma_load_4d(sb0 + C::OFF_V + q * C::TILE, &mV, bar(C::B_KVFULL), 0, h, kt * 128, b * g.S + i0 + q);
              }
            }
            kv_issued = bi + 1;
          }
          if (il == 0) {
            const int bb = u & 1;
            if (u >= 2) ok = wait_bar_warp(bar(C::B_BFREE + bb), ((u - 2) >> 1) & 1, ab);
            if (!ok) break;
            if (lane == 0) {
              const uint32_t dst = sb0 + C::OFF_BIAS + bb * C::BIAS_TILE;
              mbar_arrive_expect_tx(bar(C::B_BFULL + bb), C::BIAS_TILE);
              tma_load_3d(dst, &mBT, bar(C::B_BFULL + bb), jt * 128, kt * 128, b * g.H + h);
              tma_load_3d(dst + 16384, &mBT, bar(C::B_BFULL + bb), jt * 128 + 64, kt * 128, b * g.H + h);
            }
            ++u;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // drain copies still in flight before shared memory goes away
      if (kv_issued > 0) drain_bar(bar(C::B_KVFULL), (kv_issued - 1) & 1);
      for (int x = max(0, u - 2); x < u; ++x) drain_bar(bar(C::B_BFULL + (x & 1)), (x >> 1) & 1);
      for (int x = max(0, t - C::NQS); x < t; ++x) drain_bar(bar(C::B_QDOFULL + x % C::NQS), (x / C::NQS) & 1);
    }
  } else if (warp == C::WARP_MMA) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSS = idesc_f16(128, 128, false, false, false, false);
      constexpr uint32_t idTS = idesc_f16(128, HD, false, false, false, true);
      constexpr uint32_t idQ = idesc_f16(128, HD, false, false, true, true);
      bool ok = true;
      int t = 0;
      for (int bi = 0; bi < nblk && ok; ++bi) {
        const int i0 = s0 + bi * C::GB, nb = min(C::GB, s1 - i0);
        ok = wait_bar(bar(C::B_KVREADY), bi & 1, ab);
        if (ok && bi > 0) ok = wait_bar(bar(C::B_DKVREAD), (bi - 1) & 1, ab);
        for (int jt = 0; jt < njt && ok; ++jt) {
          for (int il = 0; il < nb && ok; ++il, ++t) {
            const int st = t % C::NQS;
            ok = wait_bar(bar(C::B_QDOREADY + st), (t / C::NQS) & 1, ab);
            if (ok && t > 0) ok = wait_bar(bar(C::B_DQREAD), (t - 1) & 1, ab);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kA = sb0 + C::OFF_K + il * C::TILE, vA = sb0 + C::OFF_V + il * C::TILE;
            const uint32_t qB = sb0 + C::OFF_Q + st * C::TILE, oB = sb0 + C::OFF_DO + st * C::TILE;
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks)
              mma_ss(tb, smem_desc(kA + ks * 32, 16, 8 * C::ROWB, C::SW), smem_desc(qB + ks * 32, 16, 8 * C::ROWB, C::SW),
                     idSS, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks)
              mma_ss(tb + 128, smem_desc(vA + ks * 32, 16, 8 * C::ROWB, C::SW),
                     smem_desc(oB + ks * 32, 16, 8 * C::ROWB, C::SW), idSS, ks > 0 ? 1u : 0u);
            mma_commit(bar(C::B_SFULL));
            ok = wait_bar(bar(C::B_PFULL), t & 1, ab);
            if (!ok) break;
            tc_fence_after();
            const uint32_t dcol = tb + 256 + il * 2 * HD;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // dV += P^T dO
              mma_ts(dcol + HD, tb + (ks >> 2) * 64 + (ks & 3) * 8, smem_desc(oB + ks * 16 * C::ROWB, 16, 8 * C::ROWB, C::SW), idTS,
                     (jt > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // dK += dS^T Q
              mma_ts(dcol, tb + 128 + (ks >> 2) * 64 + (ks & 3) * 8, smem_desc(qB + ks * 16 * C::ROWB, 16, 8 * C::ROWB, C::SW), idTS,
                     (jt > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // dQ partial = dS K
              mma_ss(tb + 96, smem_desc(sb0 + C::OFF_DS + ks * 4096, 1024, 2048, kSwizzle128B),
                     smem_desc(kA + ks * 16 * C::ROWB, 16, 8 * C::ROWB, C::SW), idQ, ks > 0 ? 1u : 0u);
            mma_commit(bar(C::B_M2DONE));
            mma_commit(bar(C::B_QDOFREE + st));
          }
        }
        mma_commit(bar(C::B_KVFREE));
      }
      mma_commit(bar(C::B_FINAL));
      drain_bar(bar(C::B_FINAL), 0);
    }
  } else {
    // ---------------------------------------------------------------- elementwise warps 0-7
    const int q = warp & 3, half = warp >> 2;
    const int kl = q * 32 + lane;  // key row of the tile = TMEM lane
    const int kg = kt * 128 + kl;
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    const float c1 = g.scale * kLog2e;
    float *maskf = reinterpret_cast<float *>(sm + C::OFF_MASK);
    const int r0 = (int)(rank * 128 / nkt), r1 = (int)((rank + 1) * 128 / nkt);
    bool ok = true;
    int t = 0, u = 0;
    auto convert_qdo = [&](int tt) -> bool {
      const int st = tt % C::NQS;
      if (!wait_bar_warp(bar(C::B_QDOFULL + st), (tt / C::NQS) & 1, ab)) return false;
      convert_to_f16(sm + C::OFF_Q + st * C::TILE, C::TILE, tid, C::NEWT);
      convert_to_f16(sm + C::OFF_DO + st * C::TILE, C::TILE, tid, C::NEWT);
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_QDOREADY + st));
      return true;
    };
    // owner side of the dQ exchange: rows [r0, r1) of every step's tile
    const int rows_max = (128 + nkt - 1) / nkt;
    const uint32_t rb_bytes = (uint32_t)(nkt * (r1 - r0) * HD * 4);
    int prev_i = 0, prev_jt = 0, red = 0;  // red = steps reduced so far
    if (tid == 0) mbar_arrive_expect_tx(bar(C::B_RFULL), rb_bytes);  // arm step 0
    auto reduce_prev = [&]() -> bool {
      if (!wait_bar_cluster_warp(bar(C::B_RFULL), red & 1, ab)) return false;
      if (tid == 0 && red + 1 < T) mbar_arrive_expect_tx(bar(C::B_RFULL), rb_bytes);  // arm the next step
      constexpr int CPR = HD / 4;
      const int items = (r1 - r0) * CPR;
      const float *rb = reinterpret_cast<const float *>(sm + C::OFF_RB);
      for (int it = tid; it < items; it += C::NEWT) {
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
          const uint2 o = make_uint2(
              (uint32_t)f32_to_bf16_rn(s4.x * g.scale) | ((uint32_t)f32_to_bf16_rn(s4.y * g.scale) << 16),
              (uint32_t)f32_to_bf16_rn(s4.z * g.scale) | ((uint32_t)f32_to_bf16_rn(s4.w * g.scale) << 16));
          *reinterpret_cast<uint2 *>(dQ + pos_row(g, b, prev_i, j) * g.H * HD + h * HD + c * 4) = o;
        }
      }
      __syncwarp();
      if (lane == 0)
        for (int r = 0; r < nkt; ++r) mbar_arrive_cluster_relaxed(mapa_shared(bar(C::B_XEMPTY), r));
      ++red;
      return true;
    };
    float acc[64];
    for (int bi = 0; bi < nblk && ok; ++bi) {
      const int i0 = s0 + bi * C::GB, nb = min(C::GB, s1 - i0);
      ok = wait_bar_warp(bar(C::B_KVFULL), bi & 1, ab);
      if (!ok) break;
      convert_to_f16(sm + C::OFF_K, nb * C::TILE, tid, C::NEWT);
      convert_to_f16(sm + C::OFF_V, nb * C::TILE, tid, C::NEWT);
      if (half == 0)
        for (int il = 0; il < nb; ++il) {
          float mv = -INFINITY;
          if (kg < g.N) mv = mask ? bf16_to_f32(mask[((int64_t)b * g.S + i0 + il) * g.N + kg]) * kLog2e : 0.f;
          maskf[il * 128 + kl] = mv;
        }
      fence_proxy_async_smem();
      mbar_arrive(bar(C::B_KVREADY));
      named_sync(1, C::NEWT);
      if (bi == 0) ok = convert_qdo(0);
      for (int jt = 0; jt < njt && ok; ++jt) {
        const int bb = u & 1;
        ok = wait_bar_warp(bar(C::B_BFULL + bb), (u >> 1) & 1, ab);
        if (!ok) break;
#pragma unroll
        for (int e = 0; e < 64; ++e) acc[e] = 0.f;
        const uint32_t brow = sb0 + C::OFF_BIAS + bb * C::BIAS_TILE + half * 16384 + kl * 128;
        for (int il = 0; il < nb; ++il, ++t) {
          const int st = t % C::NQS, i = i0 + il;
          const float mk = maskf[il * 128 + kl];
          const bool dead = (mk == -INFINITY);
          const float *sl = reinterpret_cast<const float *>(sm + C::OFF_LSE + st * 512);
          const float *sd = reinterpret_cast<const float *>(sm + C::OFF_D + st * 512);
          ok = wait_bar_warp(bar(C::B_SFULL), t & 1, ab);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int sc = 0; sc < 4; ++sc) {  // 16 query columns at a time
            const int jq0 = half * 64 + sc * 16;
            uint32_t sv[16], dv[16];
            tmem_ld16(tb + lb + jq0, sv);
            tmem_ld16(tb + lb + 128 + jq0, dv);
            tmem_wait_ld();
            uint32_t pw[8], dw[8];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int ch = sc * 2 + cc;  // 16-byte chunk (8 queries) within this query half
              uint32_t bw[4];
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(bw[0]), "=r"(bw[1]), "=r"(bw[2]), "=r"(bw[3])
                           : "r"(brow + ((ch ^ (kl & 7)) << 4)));
              float p8[8], ds8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int x = cc * 8 + e, jl = jq0 + x;
                const float bv = (e & 1) ? __uint_as_float(bw[e >> 1] & 0xffff0000u) : __uint_as_float(bw[e >> 1] << 16);
                const float arg = fmaf(__uint_as_float(sv[x]), c1, fmaf(bv, kLog2e, sl[jl] + mk));
                const float p = dead ? 0.f : ex2(arg);
                const float ds = p * (__uint_as_float(dv[x]) - sd[jl]);
                acc[sc * 16 + x] += ds;
                p8[e] = p;
                ds8[e] = ds;
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                pw[cc * 4 + e] = pack_f16x2(p8[2 * e], p8[2 * e + 1]);
                dw[cc * 4 + e] = pack_f16x2(ds8[2 * e], ds8[2 * e + 1]);
              }
              // dS (FP16) into the MN-major SW128 tile read by the dQ MMA: row kl, query chunk ch of half `half`
              const uint32_t da = sb0 + C::OFF_DS + (kl >> 3) * 2048 + half * 1024 + (kl & 7) * 128 + ((ch ^ (kl & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(da), "r"(dw[cc * 4]), "r"(dw[cc * 4 + 1]),
                           "r"(dw[cc * 4 + 2]), "r"(dw[cc * 4 + 3])
                           : "memory");
            }
            tmem_st8(tb + lb + half * 64 + sc * 8, pw);
            tmem_st8(tb + lb + 128 + half * 64 + sc * 8, dw);
          }
          fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::B_PFULL));
          if (t + 1 < T) {
            ok = convert_qdo(t + 1);
            if (!ok) break;
          }
          // ---- owner duty: reduce the previous step's dQ rows (all n partials have been pushed)
          if (t > 0) {
            ok = reduce_prev();
            if (!ok) break;
          }
          // ---- this step's dQ partial: TMEM lanes = queries, this thread has query kl, half of d
          ok = wait_bar_warp(bar(C::B_M2DONE), t & 1, ab);
          if (!ok) break;
          tc_fence_after();
          float dqv[HD / 2];
          if constexpr (HD == 32) {
            uint32_t r[16];
            tmem_ld16(tb + lb + 96 + half * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) dqv[e] = __uint_as_float(r[e]);
          } else {
            uint32_t r[8];
            tmem_ld8(tb + lb + 96 + half * 8, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) dqv[e] = __uint_as_float(r[e]);
          }
          tc_fence_before();
          mbar_arrive(bar(C::B_DQREAD));
          // every owner has finished reading its receive buffer for the previous step
          if (t > 0) ok = wait_bar_cluster_warp(bar(C::B_XEMPTY), (t - 1) & 1, ab);
          if (!ok) break;
          {
            // push row kl of this partial to its owner: rank o with o*128/n <= kl < (o+1)*128/n
            int o = (kl * nkt) >> 7;
            while (o + 1 < nkt && (int)((o + 1) * 128 / nkt) <= kl) ++o;
            while ((int)(o * 128 / nkt) > kl) --o;
            const int rl = kl - (int)(o * 128 / nkt);
            const uint32_t dst = mapa_shared(sb0 + C::OFF_RB + ((rank * rows_max + rl) * HD + half * (HD / 2)) * 4, o);
            const uint32_t rbar = mapa_shared(bar(C::B_RFULL), o);
#pragma unroll
            for (int c = 0; c < HD / 8; ++c)
              st_async_f4(dst + c * 16, dqv[4 * c], dqv[4 * c + 1], dqv[4 * c + 2], dqv[4 * c + 3], rbar);
          }
          prev_i = i;
          prev_jt = jt;
        }
        if (!ok) break;
        // ---- dBias tile (jt, kt) of this block into the supergroup partial (FP32, [k][j], owned by this CTA)
        if (kg < g.N) {
          float4 *pp = reinterpret_cast<float4 *>(
              partial + ((((int64_t)grp * g.B + b) * g.H + h) * NP + kg) * NP + jt * 128 + half * 64);
          if (bi == 0) {
#pragma unroll
            for (int c = 0; c < 16; ++c) pp[c] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
          } else {
#pragma unroll
            for (int c0 = 0; c0 < 16; c0 += 8) {
              float4 old[8];
#pragma unroll
              for (int c = 0; c < 8; ++c) old[c] = pp[c0 + c];
#pragma unroll
              for (int c = 0; c < 8; ++c)
                pp[c0 + c] = make_float4(old[c].x + acc[4 * (c0 + c)], old[c].y + acc[4 * (c0 + c) + 1],
                                         old[c].z + acc[4 * (c0 + c) + 2], old[c].w + acc[4 * (c0 + c) + 3]);
            }
          }
        }
        mbar_arrive(bar(C::B_BFREE + bb));
        ++u;
      }
      if (!ok) break;
      // ---- dK_i, dV_i of the block -> BF16 (all MMAs of the block are complete: M2DONE of its last step)
      for (int il = 0; il < nb; ++il) {
        uint32_t r[32];
        const uint32_t col = tb + lb + 256 + il * 2 * HD + half * HD;
        if constexpr (HD == 32) {
          tmem_ld32(col, r);
        } else {
          uint32_t r16[16];
          tmem_ld16(col, r16);
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = r16[e];
        }
        tmem_wait_ld();
        if (kg < g.N) {
          const float f = half == 0 ? g.scale : 1.f;
          uint16_t *out = (half == 0 ? dK : dV) + pos_row(g, b, i0 + il, kg) * g.H * HD + h * HD;
          uint32_t w[HD / 2];
#pragma unroll
          for (int c = 0; c < HD / 2; ++c)
            w[c] = (uint32_t)f32_to_bf16_rn(__uint_as_float(r[2 * c]) * f) |
                   ((uint32_t)f32_to_bf16_rn(__uint_as_float(r[2 * c + 1]) * f) << 16);
#pragma unroll
          for (int c = 0; c < HD / 8; ++c)
            reinterpret_cast<uint4 *>(out)[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DKVREAD));
    }
    if (ok && red < T) ok = reduce_prev();  // the last step's dQ rows
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tb, C::TMEM_COLS);
  }
}

// biasT[bh][k][j] = bias[bh][j][k] for j, k < N, zero in the padding up to NP.
__global__ void bias_transpose_kernel(const uint16_t *__restrict__ bias, uint16_t *__restrict__ biasT, int N,
                                      int NP) {
  __shared__ uint16_t tile[32][33];
  const int bh = blockIdx.z, j0 = blockIdx.y * 32, k0 = blockIdx.x * 32;
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

// dBias[bh][j][k] = BF16(sum over g = 0..Gp-1, in order, of partial[g][bh][k][j]).
__global__ void dbias_reduce_t_kernel(const float *__restrict__ partial, int Gp, int BH, int N, int NP,
                                      uint16_t *__restrict__ dBias) {
  __shared__ float tile[32][33];
  const int bh = blockIdx.z, k0 = blockIdx.y * 32, j0 = blockIdx.x * 32;
  const int64_t gstride = (int64_t)BH * NP * NP;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int k = k0 + r, j = j0 + threadIdx.x;
    float s = 0.f;
    if (k < N && j < N) {
      const float *p = partial + ((int64_t)bh * NP + k) * NP + j;
      s = p[0];
      for (int gi = 1; gi < Gp; ++gi) s += __ldcs(p + gi * gstride);
    }
    tile[r][threadIdx.x] = s;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int j = j0 + r, k = k0 + threadIdx.x;
    if (j < N && k < N) dBias[((int64_t)bh * N + j) * N + k] = f32_to_bf16_rn(tile[threadIdx.x][r]);
  }
}

cudaError_t launch_bias_transpose(const Dims &g, const uint16_t *bias, uint16_t *biasT, cudaStream_t stream) {
  const int NP = (g.N + 127) / 128 * 128;
  dim3 grid(NP / 32, NP / 32, g.B * g.H), block(32, 8);
  bias_transpose_kernel<<<grid, block, 0, stream>>>(bias, biasT, g.N, NP);
  return cudaGetLastError();
}

cudaError_t launch_dbias_reduce_t(const Dims &g, int Gp, const float *partial, uint16_t *dBias, cudaStream_t stream) {
  const int NP = (g.N + 127) / 128 * 128;
  dim3 grid(NP / 32, NP / 32, g.B * g.H), block(32, 8);
  dbias_reduce_t_kernel<<<grid, block, 0, stream>>>(partial, Gp, g.B * g.H, g.N, NP, dBias);
  return cudaGetLastError();
}

template <int HD>
cudaError_t launch_bwd_main_t(const Dims &g, int Gp, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                              const uint16_t *biasT, const uint16_t *mask, const float *LSE, const float *Dv,
                              const uint16_t *dO, uint16_t *dQ, uint16_t *dK, uint16_t *dV, float *partial,
                              int *status, cudaStream_t stream) {
  using C = BwdCfg<HD>;
  const int nkt = (g.N + 127) / 128, NP = nkt * 128;
  CUtensorMap mq, mk, mv, mdo, mbt;
  cudaError_t e = make_rows_map(&mq, Q, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&mk, K, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&mv, V, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&mdo, dO, g, 128);
  if (e == cudaSuccess) e = make_square_map(&mbt, biasT, NP, g.B * g.H);
  if (e != cudaSuccess) return e;
  static bool attr = false;
  if (!attr) {
    e = cudaFuncSetAttribute(bwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nkt, g.H, g.B * Gp);
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
  return cudaLaunchKernelEx(&cfg, bwd_kernel<HD>, mq, mk, mv, mdo, mbt, g, Gp, LSE, Dv, mask, dQ, dK, dV, partial,
                            status);
}

cudaError_t launch_bwd_main(const Dims &g, int Gp, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                            const uint16_t *biasT, const uint16_t *mask, const float *LSE, const float *Dv,
                            const uint16_t *dO, uint16_t *dQ, uint16_t *dK, uint16_t *dV, float *partial,
                            int *status, cudaStream_t stream) {
  if (g.d == 32)
    return launch_bwd_main_t<32>(g, Gp, Q, K, V, biasT, mask, LSE, Dv, dO, dQ, dK, dV, partial, status, stream);
  return launch_bwd_main_t<16>(g, Gp, Q, K, V, biasT, mask, LSE, Dv, dO, dQ, dK, dV, partial, status, stream);
}

int bwd_groups(const Dims &g) { return bwd_supergroups_max(g); }

// Supergroups actually launched: as many (b, h, supergroup) clusters as the
// device runs at once (one wave), within the workspace bound. Depends only on
// the shape and the GPU model, so repeated calls reduce in the same order.
template <int HD>
int bwd_groups_active_t(const Dims &g) {
  using C = BwdCfg<HD>;
  static int cache[65][9];  // [device][cluster size]
  const int nkt = (g.N + 127) / 128;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev > 64) return 1;
  int n = cache[dev][nkt];
  if (n == 0) {
    if (cudaFuncSetAttribute(bwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC) !=
        cudaSuccess)
      return 1;
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
    if (cudaOccupancyMaxActiveClusters(&n, bwd_kernel<HD>, &cfg) != cudaSuccess || n < 1) n = 1;
    cache[dev][nkt] = n;
  }
  int gp = n / (g.B * g.H);
  if (gp < 1) gp = 1;
  const int gmax = bwd_supergroups_max(g);
  return gp < gmax ? gp : gmax;
}

int bwd_groups_active(const Dims &g) { return g.d == 32 ? bwd_groups_active_t<32>(g) : bwd_groups_active_t<16>(g); }

}  // namespace triattn
