// Forward pass: tcgen05/TMEM flash-style kernel with the pair bias staged in
// shared memory and reused across the slices of a CTA.
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract): each row-slice of the pair
// tensor runs attention with a pair bias shared by all slices; the forward
// keeps BF16 outputs and, for the backward correction, a BF16 approximation of
// the output-rounding residual (O_fp32 - bf16(O)), without changing O.
//
// Work unit: batch b, head h, query tile jt (128 rows), and a group of GF
// consecutive slices. The kernel is persistent: one CTA per SM walks units
// blockIdx.x, blockIdx.x + gridDim.x, ... (units of one slice group and head
// are adjacent, so concurrent CTAs share K and V tiles in L2), with the K/V
// ring and the S buffers running on across units. For every key tile kt the bias tile
// bias[b,h,jt,kt] is brought into shared memory once as BF16 (each softmax thread
// stages its own query row, one tile ahead, double-buffered) and used for all GF slices:
//   S_i  = Q_i K_i^T           tcgen05 (BF16 x BF16 -> FP32 TMEM), M=128, N=128
//   x    = S_i*scale + bias (+ mask), m_i = running max of x  (natural units)
//   P_i  = exp2(x*log2e - m_i*log2e)   online softmax, FP32
//   O_i += P_i V_i             tcgen05 (P: FP16 in TMEM as the A operand, V: FP16)
// P is rounded to FP16 (11-bit significand) rather than BF16: a second BF16
// rounding on the output's path would add as much error as the output rounding
// itself. V is converted BF16 -> FP16 in shared memory (exact in FP16 range).
//
// Warp roles (352 threads): warps 0-7 = softmax (two threads per query row =
// TMEM lane, each owning 64 of the tile's 128 keys; the row maximum is swapped
// through shared memory), warp 8 = TMA producer, warp 9 = MMA issuer + TMEM
// owner, warp 10 = V conversion to FP16. TMEM columns: three S buffers
// [0,128) [128,256) [256,384), with P written as FP16 pairs over the columns
// each thread has already read (keys 0-63 -> cols 0-31, keys 64-127 -> cols
// 64-95 of the buffer); O_i at 384 + i*d.
// The online max is updated lazily (only when it grows by more than 2^8), and
// O is rescaled in TMEM only then. Between units the softmax warps read O out of
// TMEM (then release it to the next unit's first P.V) before they normalise and
// store it, and the next unit's first bias tile is staged during the last key tile.
#include "common.cuh"
#include "sm100.cuh"
#include "sync.cuh"
#include "tmap.cuh"

namespace triattn {
using namespace sm100;

template <int HD>
struct FwdCfg {
  static constexpr int GF = HD == 32 ? 4 : 8;  // slices per CTA
  static constexpr int NST = 4;                // K/V pipeline stages
  static constexpr int ROWB = HD * 2;          // bytes of one operand row
  static constexpr int TILE = 128 * ROWB;      // bytes of one 128-row operand tile
  static constexpr uint32_t SW = HD == 32 ? kSwizzle64B : kSwizzle32B;
  static constexpr int NMAX = TRI_ATTN_MAX_N;
  static constexpr int MAXKT = NMAX / 128;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + GF * TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_BS = OFF_V + NST * TILE;         // 2 x BF16 bias rows: 128 x 256 B (double-buffered)
  static constexpr int OFF_MASK = OFF_BS + 2 * 128 * 256;   // FP32 mask [GF][NMAX]
  static constexpr int OFF_FLAG = OFF_MASK + GF * NMAX * 4; // int [GF][MAXKT]: tile has a nonzero mask
  static constexpr int OFF_XCH = OFF_FLAG + GF * MAXKT * 4;  // row-max exchange [2][2][128] + row sums [GF][2][128]
  static constexpr int OFF_BAR = OFF_XCH + (4 + 2 * GF) * 128 * 4;
  // barrier indices
  static constexpr int B_Q = 0;
  static constexpr int B_KVFULL = 1;
  static constexpr int B_VREADY = B_KVFULL + NST;
  static constexpr int B_KVEMPTY = B_VREADY + NST;
  static constexpr int NSB = 3;                 // S buffers in TMEM
  static constexpr int B_SFULL = B_KVEMPTY + NST;
  static constexpr int B_PFULL = B_SFULL + NSB;
  static constexpr int B_SFREE = B_PFULL + NSB;
  static constexpr int B_PVDONE = B_SFREE + NSB;
  static constexpr int B_OFINAL = B_PVDONE + GF;
  static constexpr int B_OFREE = B_OFINAL + 1;  // softmax warps have read O of the unit out of TMEM
  static constexpr int B_QFREE = B_OFREE + 1;   // the unit's last S MMA has read Q
  static constexpr int B_MDRAIN = B_QFREE + 1;  // every MMA of the CTA has completed (teardown)
  static constexpr int NBAR = B_MDRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int NSOFT = 8, WARP_TMA = 8, WARP_MMA = 9, WARP_CV = 10, NTHREADS = 352;
  static constexpr uint32_t TO = NSB * 128;  // O accumulators: TO + i*d
  static_assert(TO + GF * HD <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// One work unit of the persistent forward: (b, slice group, h, query tile).
struct FwdUnit {
  int b, h, jt, i0, ng;
};

template <int HD>
__device__ __forceinline__ FwdUnit fwd_unit(const Dims &g, int u) {
  using C = FwdCfg<HD>;
  const int njt = (g.N + 127) / 128, ngroups = (g.S + C::GF - 1) / C::GF;
  FwdUnit w;
  w.jt = u % njt;
  u /= njt;
  w.h = u % g.H;
  u /= g.H;
  const int grp = u % ngroups;
  w.b = u / ngroups;
  w.i0 = grp * C::GF;
  w.ng = min(C::GF, g.S - w.i0);
  return w;
}

template <int HD>
__global__ void __launch_bounds__(FwdCfg<HD>::NTHREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
           const __grid_constant__ CUtensorMap mV, const Dims g, const uint16_t *__restrict__ bias,
           const uint16_t *__restrict__ mask, uint16_t *__restrict__ O, float *__restrict__ LSE,
           uint16_t *__restrict__ Ores, int *status) {
  using C = FwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkt = (g.N + 127) / 128;
  const int nunits = g.B * ((g.S + C::GF - 1) / C::GF) * g.H * nkt;
  auto bar = [&](int k) { return sb0 + C::OFF_BAR + 8u * (uint32_t)k; };
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_MISC);
  const Abort ab{reinterpret_cast<volatile int *>(misc + 1), status};

  if (tid == 0) {
    mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_KVFULL + s), 1);
      mbar_init(bar(C::B_VREADY + s), 1);
      mbar_init(bar(C::B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < C::NSB; ++s) {
      mbar_init(bar(C::B_SFULL + s), 1);
      mbar_init(bar(C::B_PFULL + s), 256);
      mbar_init(bar(C::B_SFREE + s), 1);
    }
    for (int s = 0; s < C::GF; ++s) mbar_init(bar(C::B_PVDONE + s), 1);
    mbar_init(bar(C::B_OFINAL), 1);
    mbar_init(bar(C::B_OFREE), 256);
    mbar_init(bar(C::B_QFREE), 1);
    mbar_init(bar(C::B_MDRAIN), 1);
    misc[1] = 0;
    fence_barrier_init();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(sb0 + C::OFF_MISC, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = misc[0];

  if (warp == C::WARP_TMA) {
    // ------------------------------------------------------------ producer
    int tg = 0, k = 0;  // tiles and units issued by this CTA
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_map(&mQ);
      tma_prefetch_map(&mK);
      tma_prefetch_map(&mV);
    }
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++k) {
      const FwdUnit w = fwd_unit<HD>(g, u);
      if (k > 0) ok = wait_bar_warp(bar(C::B_QFREE), (k - 1) & 1, ab);  // the previous unit's S MMAs read Q
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_Q), w.ng * C::TILE);
        for (int il = 0; il < w.ng; ++il)
          tma_load_4d(sb0 + C::OFF_Q + il * C::TILE, &mQ, bar(C::B_Q), 0, w.h, w.jt * 128, w.b * g.S + w.i0 + il);
      }
      const int T = nkt * w.ng;
      for (int t = 0; t < T && ok; ++t, ++tg) {
        const int st = tg % C::NST, use = tg / C::NST;
        if (use > 0) ok = wait_bar_warp(bar(C::B_KVEMPTY + st), (use - 1) & 1, ab);
        if (!ok) break;
        if (lane == 0) {
          const int kt = t / w.ng, il = t % w.ng;
          mbar_arrive_expect_tx(bar(C::B_KVFULL + st), 2 * C::TILE);
          tma_load_4d(sb0 + C::OFF_K + st * C::TILE, &mK, bar(C::B_KVFULL + st), 0, w.h, kt * 128,
                      w.b * g.S + w.i0 + il);
          tma_load_4d(sb0 + C::OFF_V + st * C::TILE, &mV, bar(C::B_KVFULL + st), 0, w.h, kt * 128,
                      w.b * g.S + w.i0 + il);
        }
      }
    }
    if (!ok && lane == 0) {
      // drain loads still in flight before the CTA's shared memory goes away
      if (k > 0) drain_bar(bar(C::B_Q), (k - 1) & 1);
      for (int t = max(0, tg - C::NST); t < tg; ++t) drain_bar(bar(C::B_KVFULL + t % C::NST), (t / C::NST) & 1);
    }
  } else if (warp == C::WARP_CV) {
    // ------------------------------------------------------------ V: BF16 -> FP16 in shared memory
    bool ok = true;
    int tg = 0;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      const int T = nkt * fwd_unit<HD>(g, u).ng;
      for (int t = 0; t < T && ok; ++t, ++tg) {
        const int st = tg % C::NST, use = tg / C::NST;
        ok = wait_bar_warp(bar(C::B_KVFULL + st), use & 1, ab);
        if (!ok) break;
        uint4 *v = reinterpret_cast<uint4 *>(sm + C::OFF_V + st * C::TILE);
        for (int e = lane; e < C::TILE / 16; e += 32) {
          uint4 x = v[e];
          x.x = bf16x2_to_f16x2(x.x);
          x.y = bf16x2_to_f16x2(x.y);
          x.z = bf16x2_to_f16x2(x.z);
          x.w = bf16x2_to_f16x2(x.w);
          v[e] = x;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_VREADY + st));
      }
    }
  } else if (warp == C::WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, true, true, false, false);
      constexpr uint32_t idPV = idesc_f16(128, HD, false, false, false, true);
      struct Pend {  // the tile whose P.V is still to be issued
        int tg, kt, il, k;
        bool last;
      };
      // O_il += P V for tile p; the first P.V of a unit first waits until the softmax warps
      // have read the previous unit's O out of TMEM
      auto issue_pv = [&](const Pend &p) -> bool {
        const int sbuf = p.tg % C::NSB, st = p.tg % C::NST;
        if (!wait_bar(bar(C::B_PFULL + sbuf), (p.tg / C::NSB) & 1, ab)) return false;
        if (!wait_bar(bar(C::B_VREADY + st), (p.tg / C::NST) & 1, ab)) return false;
        if (p.kt == 0 && p.il == 0 && p.k > 0 && !wait_bar(bar(C::B_OFREE), (p.k - 1) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t vaddr = sb0 + C::OFF_V + st * C::TILE;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tbase + C::TO + p.il * HD, tbase + sbuf * 128 + (ks >> 2) * 64 + (ks & 3) * 8,
                 smem_desc(vaddr + ks * 16 * C::ROWB, 16, 8 * C::ROWB, C::SW), idPV,
                 (p.kt > 0 || ks > 0) ? 1u : 0u);
        mma_commit(bar(C::B_SFREE + sbuf));
        mma_commit(bar(C::B_KVEMPTY + st));
        mma_commit(bar(C::B_PVDONE + p.il));
        if (p.last) mma_commit(bar(C::B_OFINAL));
        return true;
      };
      bool ok = true, pending = false;
      Pend pv{};
      int tg = 0, k = 0;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++k) {
        const int ng = fwd_unit<HD>(g, u).ng, T = nkt * ng;
        ok = wait_bar(bar(C::B_Q), k & 1, ab);
        for (int t = 0; t < T && ok; ++t, ++tg) {
          const int st = tg % C::NST, sbuf = tg % C::NSB, il = t % ng;
          ok = wait_bar(bar(C::B_KVFULL + st), (tg / C::NST) & 1, ab);
          if (ok && tg >= C::NSB) ok = wait_bar(bar(C::B_SFREE + sbuf), ((tg / C::NSB) - 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qaddr = sb0 + C::OFF_Q + il * C::TILE, kaddr = sb0 + C::OFF_K + st * C::TILE;
#pragma unroll
          for (int ks = 0; ks < HD / 16; ++ks)
            mma_ss(tbase + sbuf * 128, smem_desc(qaddr + ks * 32, 16, 8 * C::ROWB, C::SW),
                   smem_desc(kaddr + ks * 32, 16, 8 * C::ROWB, C::SW), idS, ks > 0 ? 1u : 0u);
          mma_commit(bar(C::B_SFULL + sbuf));
          if (t == T - 1) mma_commit(bar(C::B_QFREE));
          if (pending) ok = issue_pv(pv);
          pv = Pend{tg, t / ng, il, k, t == T - 1};
          pending = true;
        }
      }
      if (ok && pending) ok = issue_pv(pv);
      mma_commit(bar(C::B_MDRAIN));  // lands once every MMA issued above has completed
      drain_bar(bar(C::B_MDRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue (warps 0-7)
    // Two threads per query row: warp w handles TMEM lane quarter q = w % 4 and
    // the key half w / 4 (64 of the tile's 128 keys).
    const int q = warp & 3, half = warp >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t pair_bar = 2 + q;  // named barrier of the two warps sharing these rows
    float *maskf = reinterpret_cast<float *>(sm + C::OFF_MASK);
    int *flags = reinterpret_cast<int *>(sm + C::OFF_FLAG);
    float *xmax = reinterpret_cast<float *>(sm + C::OFF_XCH);  // [2 parities][2 halves][128 rows]
    const float2 sc2 = make_float2(g.scale, g.scale), l2e2 = make_float2(kLog2e, kLog2e);
    const uint32_t sw = row & 7;
    // bias row of a unit: rows past N reuse a valid bias row; their outputs are dropped
    auto bias_row = [&](const FwdUnit &w) {
      const int jr = min(w.jt * 128 + row, g.N - 1);
      return bias + (((int64_t)w.b * g.H + w.h) * g.N + jr) * g.N;
    };
    // this thread stages its half (64 keys) of the bias row for key tile kt into staging buffer
    // sb; keys past N get BF16 -inf, so that their scores are -inf
    auto stage_bias = [&](const uint16_t *brow, int kt, int sb) {
      const int k0 = kt * 128 + half * 64, nv = min(64, g.N - k0);
      const uint16_t *src = brow + k0;
      const uint32_t stage_row = sb0 + C::OFF_BS + sb * 32768 + row * 256;
      for (int e = max(nv, 0); e < 64; ++e)
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(stage_row + (((half * 8 + (e >> 3)) ^ sw) << 4) + (e & 7) * 2),
                     "h"((uint16_t)0xff80u));
      if (nv > 0) {
        if ((g.N & 7) == 0) {
          for (int c = 0; c < nv / 8; ++c) cp_async_16(stage_row + (((half * 8 + c) ^ sw) << 4), src + c * 8);
        } else if ((g.N & 1) == 0) {
          for (int p = 0; p < nv / 2; ++p)
            cp_async_4(stage_row + (((half * 8 + (p >> 2)) ^ sw) << 4) + (p & 3) * 4, src + 2 * p);
        } else {
          for (int e = 0; e < nv; ++e) {
            const uint16_t v = src[e];
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(stage_row + (((half * 8 + (e >> 3)) ^ sw) << 4) + (e & 7) * 2),
                         "h"(v));
          }
        }
      }
      cp_async_commit();
    };
    int pvcnt[C::GF];  // P.V commits per slice of the units before this one (PVDONE phases)
#pragma unroll
    for (int il = 0; il < C::GF; ++il) pvcnt[il] = 0;
    bool ok = true;
    int tg = 0, k = 0;
    int kb = 0;  // key tiles staged so far: tile n goes to staging buffer n & 1
    if (blockIdx.x < nunits) stage_bias(bias_row(fwd_unit<HD>(g, blockIdx.x)), 0, kb++ & 1);
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++k) {
      const FwdUnit w = fwd_unit<HD>(g, u);
      const int b = w.b, h = w.h, jt = w.jt, i0 = w.i0, ng = w.ng;
      const int j = jt * 128 + row;
      const uint16_t *brow = bias_row(w);
      // per-slice additive mask (log2 units) and per-tile "has a nonzero entry" flags
      named_sync(1, 256);  // every thread is done with the previous unit's mask rows and flags
      if (tid < C::GF * C::MAXKT) flags[tid] = 0;
      named_sync(1, 256);
      if (mask) {
        for (int il0 = 0; il0 < ng; il0 += 2) {  // two slices per memory round trip
          float v[2][C::NMAX / 256];
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int m = 0; m < C::NMAX / 256; ++m) {
              const int il = il0 + a, kk = tid + 256 * m;
              v[a][m] = (il < ng && kk < g.N) ? bf16_to_f32(mask[((int64_t)b * g.S + i0 + il) * g.N + kk]) : 0.f;
            }
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int m = 0; m < C::NMAX / 256; ++m) {
              const int il = il0 + a, kk = tid + 256 * m;
              if (il < ng && kk < nkt * 128) {
                maskf[il * C::NMAX + kk] = v[a][m];
                if (v[a][m] != 0.f) flags[il * C::MAXKT + (kk >> 7)] = 1;  // every writer stores the same value
              }
            }
        }
      }
      named_sync(1, 256);

      float m_ref[C::GF], l_sum[C::GF];  // m_ref is identical in both threads of a row; l_sum is per half
#pragma unroll
      for (int il = 0; il < C::GF; ++il) {
        m_ref[il] = -INFINITY;
        l_sum[il] = 0.f;
      }
      for (int kt = 0; kt < nkt && ok; ++kt) {
        cp_async_wait_all();  // this key tile's bias row is in staging buffer (kb - 1) & 1
        const uint32_t brow_s = sb0 + C::OFF_BS + ((kb - 1) & 1) * 32768 + row * 256;
        if (kt + 1 < nkt) {
          stage_bias(brow, kt + 1, kb++ & 1);
        } else if (u + (int)gridDim.x < nunits) {
          stage_bias(bias_row(fwd_unit<HD>(g, u + gridDim.x)), 0, kb++ & 1);  // the next unit's first tile
        }
#pragma unroll 1
        for (int il = 0; il < ng; ++il, ++tg) {
          const int sbuf = tg % C::NSB;
          ok = wait_bar_warp(bar(C::B_SFULL + sbuf), (tg / C::NSB) & 1, ab);
          if (!ok) break;
          tc_fence_after();
          const uint32_t scol = tbase + lane_base + sbuf * 128 + half * 64;
          float2 x[32];
          {
            uint32_t r[64];
            tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
            tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
            tmem_wait_ld(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
          }
          // scores in natural units: S*scale + bias (+ mask)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {  // 8 keys (16 bytes of BF16 bias) at a time
            uint32_t bw[4];
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(bw[0]), "=r"(bw[1]), "=r"(bw[2]), "=r"(bw[3])
                         : "r"(brow_s + (((half * 8 + ch) ^ sw) << 4)));
#pragma unroll
            for (int m = 0; m < 4; ++m)
              x[4 * ch + m] = __ffma2_rn(x[4 * ch + m], sc2,
                                         make_float2(__uint_as_float(bw[m] << 16), __uint_as_float(bw[m] & 0xffff0000u)));
          }
          if (flags[il * C::MAXKT + kt]) {
            const float2 *mrow = reinterpret_cast<const float2 *>(maskf + il * C::NMAX + kt * 128 + half * 64);
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = __fadd2_rn(x[e], mrow[e]);
          }
          float mloc;
          {
            float m4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) m4[c] = fmaxf(x[c].x, x[c].y);
#pragma unroll
            for (int e = 4; e < 32; ++e) m4[e & 3] = fmaxf(m4[e & 3], fmaxf(x[e].x, x[e].y));
            mloc = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          }
          // the row maximum over both key halves, exchanged through shared memory
          xmax[((tg & 1) * 2 + half) * 128 + row] = mloc;
          named_sync(pair_bar, 64);
          const float mt = fmaxf(mloc, xmax[((tg & 1) * 2 + (half ^ 1)) * 128 + row]);
          // lazy online-softmax rescale (the same decision in both threads of the row)
          float alpha = 1.f;
          bool resc = false;
          float mr = m_ref[0];
          int pvc = pvcnt[0];
#pragma unroll
          for (int qq = 1; qq < C::GF; ++qq)
            if (qq == il) {
              mr = m_ref[qq];
              pvc = pvcnt[qq];
            }
          if (kt == 0) {
            mr = mt;
          } else if (mt > mr + 8.f * kLn2) {  // grows by more than 2^8 in P
            if (mr == -INFINITY) {
              mr = mt;  // O_i and l_i are still exactly zero
            } else {
              alpha = ex2((mr - mt) * kLog2e);
              resc = true;
              mr = mt;
            }
          }
          if (__any_sync(0xffffffffu, resc)) {
            ok = wait_bar_warp(bar(C::B_PVDONE + il), (pvc + kt - 1) & 1, ab);  // P.V of key tile kt-1 done
            if (!ok) break;
            tc_fence_after();
            // this thread rescales its half of the row's O columns
            const uint32_t oaddr = tbase + lane_base + C::TO + il * HD + half * (HD / 2);
            if constexpr (HD == 32) {
              uint32_t r[16];
              tmem_ld16(oaddr, r);
              tmem_wait_ld(r);
#pragma unroll
              for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st16(oaddr, r);
            } else {
              uint32_t r[8];
              tmem_ld8(oaddr, r);
              tmem_wait_ld(r);
#pragma unroll
              for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st8(oaddr, r);
            }
          }
          const float mu = (mr == -INFINITY) ? 0.f : mr * kLog2e;
          const float2 mu2 = make_float2(-mu, -mu);
          float2 ls2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 a = __ffma2_rn(x[e], l2e2, mu2);  // (x - m) in log2 units
            const float2 pv = make_float2(ex2(a.x), ex2(a.y));
            ls2[e & 3] = __fadd2_rn(ls2[e & 3], pv);
            pk[e] = pack_f16x2(pv.x, pv.y);
          }
          const float2 lsa = __fadd2_rn(__fadd2_rn(ls2[0], ls2[1]), __fadd2_rn(ls2[2], ls2[3]));
          const float ls = lsa.x + lsa.y;
#pragma unroll
          for (int qq = 0; qq < C::GF; ++qq)
            if (qq == il) {
              m_ref[qq] = mr;
              l_sum[qq] = l_sum[qq] * alpha + ls;
            }
          // P (FP16 pairs) over this thread's own S columns: keys half*64 + [0,64) -> cols half*64 + [0,32)
          tmem_st32(scol, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::B_PFULL + sbuf));
        }
      }
      if (!ok) break;
#pragma unroll
      for (int il = 0; il < C::GF; ++il)
        if (il < ng) pvcnt[il] += nkt;
      // epilogue: read O of the unit out of TMEM and release it, then O = acc / l -> BF16, residual, LSE
      ok = wait_bar_warp(bar(C::B_OFINAL), k & 1, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t oacc[C::GF][HD / 2] = {};
#pragma unroll
      for (int il = 0; il < C::GF; ++il) {
        if (il < ng) {
          const uint32_t oaddr = tbase + lane_base + C::TO + il * HD + half * (HD / 2);
          if constexpr (HD == 32) {
            tmem_ld16(oaddr, oacc[il]);
          } else {
            tmem_ld8(oaddr, oacc[il]);
          }
        }
      }
      tmem_wait_ld(oacc);
      tc_fence_before();
      mbar_arrive(bar(C::B_OFREE));
      float *xl = reinterpret_cast<float *>(sm + C::OFF_XCH) + 4 * 128;  // [GF][2 halves][128 rows]
#pragma unroll
      for (int qq = 0; qq < C::GF; ++qq) xl[(qq * 2 + half) * 128 + row] = l_sum[qq];
      named_sync(pair_bar, 64);
#pragma unroll
      for (int il = 0; il < C::GF; ++il) {
        if (il >= ng) continue;
        const float lsum = xl[(il * 2 + 0) * 128 + row] + xl[(il * 2 + 1) * 128 + row];
        if (j < g.N) {
          const int i = i0 + il;
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
          uint32_t ob[HD / 4], rb[HD / 4];
#pragma unroll
          for (int c = 0; c < HD / 4; ++c) {
            const float o0 = __uint_as_float(oacc[il][2 * c]) * inv, o1 = __uint_as_float(oacc[il][2 * c + 1]) * inv;
            const uint16_t a0 = f32_to_bf16_rn(o0), a1 = f32_to_bf16_rn(o1);
            ob[c] = (uint32_t)a0 | ((uint32_t)a1 << 16);
            rb[c] = (uint32_t)f32_to_bf16_rn(o0 - bf16_to_f32(a0)) |
                    ((uint32_t)f32_to_bf16_rn(o1 - bf16_to_f32(a1)) << 16);
          }
          const int64_t off = pos_row(g, b, i, j) * g.H * HD + (int64_t)h * HD + half * (HD / 2);
          // this thread's half row: 32 bytes (d = 32) or 16 bytes (d = 16), one store each
          if constexpr (HD == 32) {
            asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(O + off), "r"(ob[0]), "r"(ob[1]),
                         "r"(ob[2]), "r"(ob[3]), "r"(ob[4]), "r"(ob[5]), "r"(ob[6]), "r"(ob[7])
                         : "memory");
            if (Ores)
              asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(Ores + off), "r"(rb[0]),
                           "r"(rb[1]), "r"(rb[2]), "r"(rb[3]), "r"(rb[4]), "r"(rb[5]), "r"(rb[6]), "r"(rb[7])
                           : "memory");
          } else {
            *reinterpret_cast<uint4 *>(O + off) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
            if (Ores) *reinterpret_cast<uint4 *>(Ores + off) = make_uint4(rb[0], rb[1], rb[2], rb[3]);
          }
          if (half == 0)
            LSE[(((int64_t)b * g.S + i) * g.H + h) * g.N + j] =
                lsum > 0.f ? m_ref[il] + __log2f(lsum) * kLn2 : -INFINITY;
        }
      }
    }
    cp_async_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int HD>
cudaError_t launch_fwd_t(const Dims &g, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                         const uint16_t *bias, const uint16_t *mask, uint16_t *O, float *LSE, uint16_t *Ores,
                         int *status, cudaStream_t stream) {
  using C = FwdCfg<HD>;
  CUtensorMap mq, mk, mv;
  cudaError_t e = make_rows_map(&mq, Q, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&mk, K, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&mv, V, g, 128);
  if (e != cudaSuccess) return e;
  static bool attr = false;
  if (!attr) {
    e = cudaFuncSetAttribute(fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  // persistent: one CTA per resident slot, each walking units blockIdx.x, +gridDim.x, ...
  static int slots[65];
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev > 64) return cudaErrorInvalidDevice;
  if (slots[dev] == 0) {
    int nsm = 0, per = 0;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fwd_kernel<HD>, C::NTHREADS, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    slots[dev] = max(1, nsm * per);
  }
  const int nunits = g.B * ((g.S + C::GF - 1) / C::GF) * g.H * ((g.N + 127) / 128);
  const int grid = min(nunits, slots[dev]);
  fwd_kernel<HD><<<grid, C::NTHREADS, C::SMEM_ALLOC, stream>>>(mq, mk, mv, g, bias, mask, O, LSE, Ores, status);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const Dims &g, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                       const uint16_t *bias, const uint16_t *mask, uint16_t *O, float *LSE, uint16_t *Ores,
                       int *status, cudaStream_t stream) {
  if (g.d == 32) return launch_fwd_t<32>(g, Q, K, V, bias, mask, O, LSE, Ores, status, stream);
  return launch_fwd_t<16>(g, Q, K, V, bias, mask, O, LSE, Ores, status, stream);
}

}  // namespace triattn
