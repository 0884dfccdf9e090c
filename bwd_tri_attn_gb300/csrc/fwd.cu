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
// ring, the bias and mask buffers and the S buffers running on across units.
// For every key tile kt the bias tile bias[b,h,jt,kt] is brought into shared
// memory once (BF16, by TMA) and used for all GF slices:
//   S_i  = Q_i K_i^T           tcgen05 (BF16 x BF16 -> FP32 TMEM), M=128, N=128
//   x    = S_i*scale + bias (+ mask), m_i = running max of x  (natural units)
//   P_i  = exp2(x*log2e - m_i*log2e)   online softmax, FP32
//   O_i += P_i V_i             tcgen05 (P: FP16 in TMEM as the A operand, V: FP16)
// P is rounded to FP16 (11-bit significand) rather than BF16: a second BF16
// rounding on the output's path would add as much error as the output rounding
// itself. V is converted BF16 -> FP16 in shared memory by the softmax threads, a
// slice of the tile each, before they hand P over; every (b, i, h) block of V is
// first multiplied by the power of two 2^sv that brings its largest magnitude into
// [2^14, 2^15) (exact, and FP16 then holds every entry within 2^-31 of that largest
// one at full precision), and O is multiplied by 2^-sv in the epilogue. A pre-pass
// (fwd_vscale_kernel) finds sv and leaves it in LSE[b, i, h, 128 jt] for every query
// tile jt: the one LSE slot per work unit that the unit reads at its start and only
// overwrites, with the log-sum-exp, at its end.
//
// Warp roles (384 threads): warp 0 = producer (TMA for Q, K, V and the bias
// tiles, bulk copies of the mask rows and their per-tile "nonzero" flags),
// warp 1 = P.V issuer + TMEM owner, warp 2 = S issuer, warp 3 only donates
// registers; warps 4-11 = softmax, one thread per query row (TMEM lane) over all
// 128 keys of a tile: softmax warpgroup 0 (warps 4-7) takes the slices
// il = 0, 2, ... and softmax warpgroup 1 (warps 8-11) the slices il = 1, 3, ...
// of every key tile, so the two work on different S tiles at once and never
// wait on each other inside a key tile (setmaxnreg: 216 per softmax thread).
// TMEM columns: three S buffers [0,128) [128,256) [256,384), with P written as
// FP16 pairs over the columns the thread has already read (keys 0-63 -> cols
// 0-31, keys 64-127 -> cols 64-95 of the buffer); O_i at 384 + i*d.
// The online max is updated lazily (only when it grows by more than 2^8), and
// O is rescaled in TMEM only then, after the slice's previous P.V has completed. Between units the softmax warps read O out of
// TMEM (then release it to the next unit's first P.V) before they normalise and
// store it.
//
// Shapes with N not a multiple of 8 (bias rows not 16-byte aligned, so no TMA
// view) take a fallback where each softmax thread stages its own bias row one
// key tile ahead with cp.async and the producer copies the mask rows lane by lane.
#include "common.cuh"
#include "launch.cuh"
#include "plan.cuh"
#include "sm100.cuh"
#include "sync.cuh"
#include "tmap.cuh"

#include <string.h>

namespace triattn {
using namespace sm100;

template <int HD>
struct FwdCfg {
  static constexpr int GF = 4;  // slices per work unit (8 at d = 16 measured 3 % slower)
  static constexpr int NSB = 3;                // S buffers in TMEM: tile tg uses buffer tg % 3
  static constexpr int NST = 6;                // K/V pipeline stages: tile tg uses stage tg % 6
  static constexpr int ROWB = HD * 2;          // bytes of one operand row
  static constexpr int TILE = 128 * ROWB;      // bytes of one 128-row operand tile
  static constexpr uint32_t SW = HD == 32 ? kSwizzle64B : kSwizzle32B;
  static constexpr int NMAX = TRI_ATTN_MAX_N;
  static constexpr int MAXKT = NMAX / 128;
  static constexpr int BTILE = 128 * 256;                   // BF16 bias tile: [2 halves][128 rows][128 B], SW128
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + GF * TILE;
  static constexpr int OFF_V = OFF_K + NST * TILE;
  static constexpr int OFF_BS = OFF_V + NST * TILE;         // 2 bias tiles (double-buffered by key tile)
  static constexpr int OFF_MASK = OFF_BS + 2 * BTILE;       // 2 x BF16 mask rows [GF][NMAX] (by unit)
  static constexpr int OFF_FLAG = OFF_MASK + 2 * GF * NMAX * 2;  // 2 x int [GF][MAXKT]: tile has a nonzero mask entry
  static constexpr int OFF_BAR = OFF_FLAG + 2 * GF * MAXKT * 4;
  // barrier indices
  static constexpr int B_Q = 0;                 // [GF] Q tile of slice il landed
  static constexpr int B_KVFULL = B_Q + GF;
  static constexpr int B_KVEMPTY = B_KVFULL + NST;  // the stage's P.V has completed
  static constexpr int B_SFULL = B_KVEMPTY + NST;
  static constexpr int B_PFULL = B_SFULL + NSB;  // P written and this tile's V converted
  static constexpr int B_TDONE = B_PFULL + NSB;  // the buffer's P.V has completed: the S buffer is free
  static constexpr int B_OFINAL = B_TDONE + NSB;  // [2] the warpgroup's O accumulators of the unit are final
  static constexpr int B_OFREE = B_OFINAL + 2;    // [2] the warpgroup has read its O of the unit out of TMEM
  static constexpr int B_QFREE = B_OFREE + 2;     // [GF] the unit's last S MMA of slice il has read Q_il
  static constexpr int B_MDRAIN = B_QFREE + GF;   // [2] every MMA of the S / P.V issuer has completed (teardown)
  static constexpr int B_PVDONE = B_MDRAIN + 2;   // [GF] a P.V of slice il has completed (one phase per P.V)
  static constexpr int B_BFULL = B_PVDONE + GF;  // [2] bias tile landed
  static constexpr int B_BFREE = B_BFULL + 2;   // [2] every slice of its key tile is done with it
  static constexpr int B_MFULL = B_BFREE + 2;   // [2] mask rows of a unit landed
  static constexpr int B_MFREE = B_MFULL + 2;   // [2] the unit is done with them
  static constexpr int B_MREADY = B_MFREE + 2;  // [2] mask rows and their tile flags in place
  static constexpr int B_BSTAGE = B_MREADY + 2;  // (N % 8 != 0) both warpgroups staged their half of a bias tile
  static constexpr int NBAR = B_BSTAGE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  // the control warps take the lowest warp indices (warpgroup 0): warp schedulers favour low-index
  // warps, and these warps' short instruction sequences gate everyone else's progress
  static constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_S = 2, WARP_SOFT0 = 4, NTHREADS = 384;  // warp 3: donor
  // setmaxnreg split: the softmax warpgroups take registers from the third warpgroup (per SMSP:
  // two softmax warps and one other warp share 16K registers)
  static constexpr uint32_t REG_LAUNCH = 168, REG_SOFT = 216, REG_OTHER = 72;
  static_assert(256 * REG_SOFT + (NTHREADS - 256) * REG_OTHER == NTHREADS * REG_LAUNCH, "register split");
  static constexpr uint32_t TO = NSB * 128;  // O accumulators: TO + i*d
  static_assert(TO + GF * HD <= TMEM_COLS, "TMEM budget");
  static_assert(OFF_BS % 1024 == 0, "SW128 bias tiles need 1 KB alignment");
  static_assert(TILE % (16 * 128) == 0, "V conversion: whole 16-byte chunks per softmax thread");
  static_assert(GF % 2 == 0, "slices split evenly over the two softmax warpgroups");
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

// Scale exponent sv of every (b, i, h) block of V (one CTA each, heads fastest), written into
// the LSE slot of each work unit of that block.
template <int HD, int NODE>
__global__ void __launch_bounds__(256) fwd_vscale_kernel(const Dims g, const uint4 *__restrict__ V,
                                                         int *__restrict__ lse_bits) {
  __shared__ int red[8];
  constexpr int CPH = HD / 8, PPP = 256 / CPH;
  const int h = blockIdx.x, bi = blockIdx.y, b = bi / g.S, i = bi - b * g.S;
  const int c = threadIdx.x % CPH, cpp = g.H * CPH;
  uint32_t m = 0;
  for (int j = threadIdx.x / CPH; j < g.N; j += PPP)
    m = exp_max4(m, ld_stream(V + pos_row(g, b, i, j, NODE) * cpp + h * CPH + c));
  const int s = scale_exp(block_max<256>(bf16x2_exp_final(m), red), kTargetQK);
  int *row = lse_bits + ((int64_t)bi * g.H + h) * g.N;
  for (int jt = threadIdx.x; jt * 128 < g.N; jt += 256) row[jt * 128] = s;
}

template <int HD, int NODE>
__global__ void __launch_bounds__(FwdCfg<HD>::NTHREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
           const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mB, const Dims g,
           const uint16_t *__restrict__ bias, const uint16_t *__restrict__ mask, uint16_t *__restrict__ O,
           float *__restrict__ LSE, uint16_t *__restrict__ Ores, int *status) {
  using C = FwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb0 = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkt = (g.N + 127) / 128;
  const int nunits = g.B * ((g.S + C::GF - 1) / C::GF) * g.H * nkt;
  const bool tma_bias = (g.N & 7) == 0;  // bias rows 16-byte aligned: TMA tiles; else per-thread staging
  auto bar = [&](int k) { return sb0 + C::OFF_BAR + 8u * (uint32_t)k; };
  volatile uint32_t *misc = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_MISC);
  const Abort ab{reinterpret_cast<volatile int *>(misc + 1), status};

  if (tid == 0) {
    for (int s = 0; s < C::GF; ++s) {
      mbar_init(bar(C::B_Q + s), 1);
      mbar_init(bar(C::B_QFREE + s), 1);
      mbar_init(bar(C::B_PVDONE + s), 1);
    }
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_KVFULL + s), 1);
      mbar_init(bar(C::B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < C::NSB; ++s) {
      mbar_init(bar(C::B_SFULL + s), 1);
      mbar_init(bar(C::B_PFULL + s), 128);  // the warpgroup that owns the tile
      mbar_init(bar(C::B_TDONE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_MDRAIN + s), 1);
      mbar_init(bar(C::B_OFINAL + s), 1);
      mbar_init(bar(C::B_OFREE + s), 128);
      mbar_init(bar(C::B_BFULL + s), 1);
      mbar_init(bar(C::B_BFREE + s), 256);
      mbar_init(bar(C::B_MFULL + s), 1);
      mbar_init(bar(C::B_MFREE + s), 256);
      mbar_init(bar(C::B_MREADY + s), 1);
    }
    mbar_init(bar(C::B_BSTAGE), 256);
    misc[1] = 0;
    fence_barrier_init();
  }
  if (mask && (g.N & 127) != 0) {
    // keys in [N, nkt*128) of both mask buffers read as 0 (the copies never write them)
    uint16_t *mk = reinterpret_cast<uint16_t *>(sm + C::OFF_MASK);
    const int tail = nkt * 128 - g.N;
    for (int x = tid; x < 2 * C::GF * tail; x += C::NTHREADS) mk[(x / tail) * C::NMAX + g.N + x % tail] = 0;
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
    reg_dealloc<C::REG_OTHER>();
    int tg = 0, k = 0, kb = 0;  // tiles, units and bias tiles issued by this CTA
    uint32_t qcur = 0;          // Q buffers whose phase of the current unit has been started
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_map(&mQ);
      tma_prefetch_map(&mK);
      tma_prefetch_map(&mV);
      if (tma_bias) tma_prefetch_map(&mB);
    }
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++k) {
      const FwdUnit w = fwd_unit<HD>(g, u);
      qcur = 0;
      // Q buffers of slices the unit does not have complete their phase at once (every buffer
      // goes through one phase per unit); the others are loaded with the unit's first key tile
      for (int il = w.ng; il < C::GF && ok; ++il) {
        if (k > 0) ok = wait_bar_warp(bar(C::B_QFREE + il), (k - 1) & 1, ab);
        if (ok && lane == 0) mbar_arrive(bar(C::B_Q + il));
        if (ok) qcur |= 1u << il;
      }
      if (!ok) break;
      if (mask) {  // the unit's mask rows into buffer k & 1 (free once unit k - 2 is done)
        if (k >= 2) ok = wait_bar_warp(bar(C::B_MFREE + (k & 1)), ((k - 2) >> 1) & 1, ab);
        if (!ok) break;
        const uint32_t mdst = sb0 + C::OFF_MASK + (k & 1) * (C::GF * C::NMAX * 2);
        const uint16_t *msrc = mask + ((int64_t)w.b * g.S + w.i0) * g.N;
        if (tma_bias) {
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_MFULL + (k & 1)), w.ng * g.N * 2);
            for (int il = 0; il < w.ng; ++il)
              bulk_load(mdst + il * C::NMAX * 2, msrc + (int64_t)il * g.N, g.N * 2, bar(C::B_MFULL + (k & 1)));
          }
        } else {
          uint16_t *md = reinterpret_cast<uint16_t *>(sm + C::OFF_MASK) + (k & 1) * (C::GF * C::NMAX);
          for (int il = 0; il < w.ng; ++il)
            for (int e0 = lane; e0 < g.N; e0 += 256) {  // eight loads in flight per lane
              uint16_t v[8];
#pragma unroll
              for (int m = 0; m < 8; ++m) v[m] = e0 + 32 * m < g.N ? msrc[(int64_t)il * g.N + e0 + 32 * m] : 0;
#pragma unroll
              for (int m = 0; m < 8; ++m)
                if (e0 + 32 * m < g.N) md[il * C::NMAX + e0 + 32 * m] = v[m];
            }
        }
        // per (slice, key tile): does the tile hold a nonzero mask entry (read once here, so that the
        // softmax threads add mask values only where they change something)
        if (tma_bias) ok = wait_bar_warp(bar(C::B_MFULL + (k & 1)), (k >> 1) & 1, ab);
        if (!ok) break;
        __syncwarp();
        const uint16_t *mrows = reinterpret_cast<const uint16_t *>(sm + C::OFF_MASK) + (k & 1) * (C::GF * C::NMAX);
        int *fl = reinterpret_cast<int *>(sm + C::OFF_FLAG) + (k & 1) * (C::GF * C::MAXKT);
        for (int x = lane; x < w.ng * nkt; x += 32) {
          const int il = x / nkt, kt = x % nkt;
          const uint4 *mr = reinterpret_cast<const uint4 *>(mrows + il * C::NMAX + kt * 128);
          uint32_t any = 0;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint4 v = mr[c];
            any |= v.x | v.y | v.z | v.w;
          }
          fl[il * C::MAXKT + kt] = (any & 0x7fff7fffu) != 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_MREADY + (k & 1)));
      }
      const int T = nkt * w.ng;
      for (int t = 0; t < T && ok; ++t, ++tg) {
        if (tma_bias && t % w.ng == 0) {  // bias tile (jt, kt) into buffer kb & 1 (free once tile kb - 2 is done)
          if (kb >= 2) ok = wait_bar_warp(bar(C::B_BFREE + (kb & 1)), ((kb - 2) >> 1) & 1, ab);
          if (!ok) break;
          if (lane == 0) {
            const int kt = t / w.ng;
            const uint32_t dst = sb0 + C::OFF_BS + (kb & 1) * C::BTILE;
            mbar_arrive_expect_tx(bar(C::B_BFULL + (kb & 1)), C::BTILE);
            tma_load_3d(dst, &mB, bar(C::B_BFULL + (kb & 1)), kt * 128, w.jt * 128, w.b * g.H + w.h);
            tma_load_3d(dst + C::BTILE / 2, &mB, bar(C::B_BFULL + (kb & 1)), kt * 128 + 64, w.jt * 128,
                        w.b * g.H + w.h);
          }
          ++kb;
        }
        if (t < w.ng) {  // Q_il, once the previous unit's last S MMA of slice il has read the buffer
          if (k > 0) ok = wait_bar_warp(bar(C::B_QFREE + t), (k - 1) & 1, ab);
          if (!ok) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(C::B_Q + t), C::TILE);
            load_rows(sb0 + C::OFF_Q + t * C::TILE, &mQ, bar(C::B_Q + t), NODE, w.h, w.b, g.S, w.i0 + t, w.jt * 128);
          }
          qcur |= 1u << t;
        }
        const int st = tg % C::NST, use = tg / C::NST;
        if (use > 0) ok = wait_bar_warp(bar(C::B_KVEMPTY + st), (use - 1) & 1, ab);
        if (!ok) break;
        if (lane == 0) {
          const int kt = t / w.ng, il = t % w.ng;
          mbar_arrive_expect_tx(bar(C::B_KVFULL + st), 2 * C::TILE);
          load_rows(sb0 + C::OFF_K + st * C::TILE, &mK, bar(C::B_KVFULL + st), NODE, w.h, w.b, g.S, w.i0 + il, kt * 128);
          load_rows(sb0 + C::OFF_V + st * C::TILE, &mV, bar(C::B_KVFULL + st), NODE, w.h, w.b, g.S, w.i0 + il, kt * 128);
        }
      }
    }
    if (!ok && lane == 0) {
      // drain copies still in flight before the CTA's shared memory goes away
      for (int il = 0; il < C::GF; ++il) {
        if ((qcur >> il) & 1) {
          drain_bar(bar(C::B_Q + il), k & 1);
        } else if (k > 0) {
          drain_bar(bar(C::B_Q + il), (k - 1) & 1);
        }
      }
      if (mask && tma_bias && k > 0) drain_bar(bar(C::B_MFULL + ((k - 1) & 1)), ((k - 1) >> 1) & 1);
      for (int x = max(0, kb - 2); x < kb; ++x) drain_bar(bar(C::B_BFULL + (x & 1)), (x >> 1) & 1);
      for (int t = max(0, tg - C::NST); t < tg; ++t) drain_bar(bar(C::B_KVFULL + t % C::NST), (t / C::NST) & 1);
    }
  } else if (warp == C::WARP_MMA || warp == C::WARP_S) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 2 issues S = Q K^T, warp 1 P.V, each walking the CTA's tiles in order (units
    // blockIdx.x, +gridDim.x, ...; in a unit key tile kt, then slice il) with blocking waits on
    // exactly the barriers that gate its next MMA. Each warp runs converged; elect.sync picks
    // the lane that issues. A commit covers the MMAs of the issuing thread only, so every
    // barrier below is committed by the warp whose MMAs it certifies.
    reg_dealloc<C::REG_OTHER>();
    constexpr uint32_t idS = idesc_f16(128, 128, true, true, false, false);
    constexpr uint32_t idPV = idesc_f16(128, HD, false, false, false, true);
    // descriptor bases: the start-address field is (address >> 4) in the low bits, so an operand
    // at base + off has descriptor base_desc + (off >> 4) (addresses stay below 256 KB)
    const uint64_t dq0 = smem_desc(sb0 + C::OFF_Q, 16, 8 * C::ROWB, C::SW);
    const uint64_t dk0 = smem_desc(sb0 + C::OFF_K, 16, 8 * C::ROWB, C::SW);
    const uint64_t dv0 = smem_desc(sb0 + C::OFF_V, 16, 8 * C::ROWB, C::SW);
    const bool is_s = warp == C::WARP_S;
    bool ok = true;
    int tg = 0, k = 0;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++k) {
      const int ng = fwd_unit<HD>(g, u).ng, T = nkt * ng;
      int il = 0, kt = 0;
      for (int t = 0; t < T && ok; ++t, ++tg) {
        const int sbuf = tg % C::NSB, st = tg % C::NST;
        if (is_s) {
          // S into buffer tg % NSB: Q_il and the tile's K landed, the buffer's previous P.V done
          ok = wait_bar_warp(bar(C::B_Q + il), k & 1, ab) && wait_bar_warp(bar(C::B_KVFULL + st), (tg / C::NST) & 1, ab) &&
               (tg < C::NSB || wait_bar_warp(bar(C::B_TDONE + sbuf), ((tg / C::NSB) - 1) & 1, ab));
          if (!ok) break;
          tc_fence_after();
          const uint64_t dq = dq0 + (uint64_t)((il * C::TILE) >> 4), dk = dk0 + (uint64_t)((st * C::TILE) >> 4);
          mma_ss_e(tbase + sbuf * 128, dq, dk, idS, 0u);
#pragma unroll
          for (int ks = 1; ks < HD / 16; ++ks) mma_ss_e(tbase + sbuf * 128, dq + 2 * ks, dk + 2 * ks, idS, 1u);
          mma_commit_e(bar(C::B_SFULL + sbuf));
          if (t >= T - ng) mma_commit_e(bar(C::B_QFREE + il));  // the unit's last S of slice il
          if (t == T - 1)
            for (int q = ng; q < C::GF; ++q) mma_commit_e(bar(C::B_QFREE + q));
        } else {
          // O_il += P V: P written and V converted (PFULL); a unit's first P.V of a slice overwrites
          // the accumulator, so the previous unit's O must have been read out (OFREE)
          ok = wait_bar_warp(bar(C::B_PFULL + sbuf), (tg / C::NSB) & 1, ab) &&
               (kt > 0 || k == 0 || wait_bar_warp(bar(C::B_OFREE + (il & 1)), (k - 1) & 1, ab));
          if (!ok) break;
          tc_fence_after();
          const uint64_t dv = dv0 + (uint64_t)((st * C::TILE) >> 4);
          const uint32_t dO = tbase + C::TO + il * HD, aP = tbase + sbuf * 128;
          // K step ks: P columns (ks >> 2) * 64 + (ks & 3) * 8, V rows 16 ks
          mma_ts_x8_e<0, 8, 16, 24, 64, 72, 80, 88>(dO, aP, dv, (uint64_t)((16 * C::ROWB) >> 4), idPV, kt > 0 ? 1u : 0u);
          mma_commit_e(bar(C::B_TDONE + sbuf));
          mma_commit_e(bar(C::B_KVEMPTY + st));
          mma_commit_e(bar(C::B_PVDONE + il));
          // the warpgroup's O is final after the P.V of its last slice in the last key tile; a
          // warpgroup without slices in this unit is released with the unit's last P.V
          if (kt == nkt - 1 && il + 2 >= ng) mma_commit_e(bar(C::B_OFINAL + (il & 1)));
          if (t == T - 1 && ng == 1) mma_commit_e(bar(C::B_OFINAL + 1));
        }
        if (++il == ng) {
          il = 0;
          ++kt;
        }
      }
    }
    const uint32_t drain = bar(C::B_MDRAIN + (is_s ? 1 : 0));
    mma_commit_e(drain);  // lands once every MMA this warp issued has completed
    if (lane == 0) drain_bar(drain, 0);
    __syncwarp();
  } else if (warp >= C::WARP_SOFT0) {
    // ------------------------------------------------------------ softmax / epilogue (warps 4-11)
    reg_alloc<C::REG_SOFT>();
    // One thread per query row (TMEM lane); warpgroup wg = warp / 4 takes the slices
    // il = wg, wg + 2, ... of every key tile, so the two warpgroups work on different
    // S tiles at the same time and never wait on each other within a key tile.
    constexpr int NL = C::GF / 2;  // slices per warpgroup
    const int q = warp & 3, wg = (warp - C::WARP_SOFT0) >> 2, wtid = tid & 127;
    const int row = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const float2 sc2 = make_float2(g.scale, g.scale), l2e2 = make_float2(kLog2e, kLog2e);
    const uint32_t sw = row & 7;
    // this thread's row of a bias tile: [half][row][128 B], 16-byte chunk c at ((c ^ (row & 7)) << 4)
    const uint32_t brow_off = (uint32_t)(row * 128);
    // fallback staging (N not a multiple of 8): warpgroup wg copies key half wg of its rows of key
    // tile kt into bias buffer sb, keys past N as BF16 -inf; rows past N reuse a valid bias row
    auto stage_bias = [&](const FwdUnit &w, int kt, int sb) {
      const int jr = min(w.jt * 128 + row, g.N - 1);
      const uint16_t *src = bias + (((int64_t)w.b * g.H + w.h) * g.N + jr) * g.N + kt * 128 + wg * 64;
      const int nv = min(64, g.N - (kt * 128 + wg * 64));
      const uint32_t dst = sb0 + C::OFF_BS + sb * C::BTILE + wg * (C::BTILE / 2) + brow_off;
      for (int e = max(nv, 0); e < 64; ++e)
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(dst + (((e >> 3) ^ sw) << 4) + (e & 7) * 2), "h"((uint16_t)0xff80u));
      if ((g.N & 1) == 0) {
        for (int p = 0; p < nv / 2; ++p) cp_async_4(dst + (((p >> 2) ^ sw) << 4) + (p & 3) * 4, src + 2 * p);
      } else {
        for (int e = 0; e < nv; ++e) {
          const uint16_t v = src[e];
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(dst + (((e >> 3) ^ sw) << 4) + (e & 7) * 2), "h"(v));
        }
      }
      cp_async_commit();
    };
    bool ok = true;
    int tgu = 0, k = 0;  // tiles of the units before this one, units done
    int kb = 0;          // key tiles of bias used so far: tile n lives in bias buffer n & 1
    int pvc[NL];         // P.V of this warpgroup's slice slots in the units before this one
#pragma unroll
    for (int s = 0; s < NL; ++s) pvc[s] = 0;
    if (!tma_bias && blockIdx.x < nunits) stage_bias(fwd_unit<HD>(g, blockIdx.x), 0, 0);
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++k) {
      const FwdUnit w = fwd_unit<HD>(g, u);
      const int b = w.b, h = w.h, jt = w.jt, i0 = w.i0, ng = w.ng;
      const int j = jt * 128 + row;
      const uint16_t *mk = reinterpret_cast<const uint16_t *>(sm + C::OFF_MASK) + (k & 1) * (C::GF * C::NMAX);
      const int *flags = reinterpret_cast<const int *>(sm + C::OFF_FLAG) + (k & 1) * (C::GF * C::MAXKT);
      // V scale of this warpgroup's slices (their LSE slots of this unit; see fwd_vscale_kernel)
      float vsc[NL], vinv[NL];
#pragma unroll
      for (int s = 0; s < NL; ++s) {
        const int il = wg + 2 * s, e = il < ng ? reinterpret_cast<const int *>(LSE)[(((int64_t)b * g.S + i0 + il) * g.H + h) * g.N + jt * 128] : 0;
        vsc[s] = exp2i(e);
        vinv[s] = exp2i(-e);
      }
      if (mask) ok = wait_bar_warp(bar(C::B_MREADY + (k & 1)), (k >> 1) & 1, ab);
      if (!ok) break;

      float m_ref[NL], l_sum[NL];
#pragma unroll
      for (int s = 0; s < NL; ++s) {
        m_ref[s] = -INFINITY;
        l_sum[s] = 0.f;
      }
      for (int kt = 0; kt < nkt && ok; ++kt, ++kb) {
        if (tma_bias) {
          ok = wait_bar_warp(bar(C::B_BFULL + (kb & 1)), (kb >> 1) & 1, ab);
          if (!ok) break;
        } else {
          cp_async_wait_all();  // this warpgroup's half of the tile is in buffer kb & 1
          // and the other half; every thread is done with tile kb - 1. A bounded wait: if the other
          // warpgroup has given up (its own wait expired) it arrives no more, and this one leaves
          // through the abort flag instead of hanging.
          mbar_arrive(bar(C::B_BSTAGE));
          ok = wait_bar_warp(bar(C::B_BSTAGE), kb & 1, ab);
          if (!ok) break;
          if (kt + 1 < nkt) {
            stage_bias(w, kt + 1, (kb + 1) & 1);
          } else if (u + (int)gridDim.x < nunits) {
            stage_bias(fwd_unit<HD>(g, u + gridDim.x), 0, (kb + 1) & 1);  // the next unit's first tile
          }
        }
        const uint32_t brow_s = sb0 + C::OFF_BS + (kb & 1) * C::BTILE + brow_off;
        const int nvalid = g.N - kt * 128;  // keys past N in the last key tile get score -inf
#pragma unroll 1
        for (int il = wg; il < ng; il += 2) {
          const int tg = tgu + kt * ng + il, sbuf = tg % C::NSB, sl = il >> 1;
          ok = wait_bar_warp(bar(C::B_SFULL + sbuf), (tg / C::NSB) & 1, ab);
          if (!ok) break;
          tc_fence_after();
          const uint32_t scol = tbase + lane_base + sbuf * 128;
          float2 x[64];
          {
            uint32_t r[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(scol + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
            tmem_wait_ld(r);
#pragma unroll
            for (int e = 0; e < 64; ++e) x[e] = make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
          }
          // scores in natural units: S*scale + bias (+ mask); the bias chunks (8 keys, 16 bytes of
          // BF16) are loaded four ahead of their use
          {
            uint32_t bw[4][4];
            auto bias_ld = [&](int ch, uint32_t(&w)[4]) {
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                           : "r"(brow_s + (ch >> 3) * (C::BTILE / 2) + (((ch & 7) ^ sw) << 4)));
            };
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) bias_ld(ch, bw[ch]);
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
              uint32_t cur[4];
#pragma unroll
              for (int m = 0; m < 4; ++m) cur[m] = bw[ch & 3][m];
              if (ch + 4 < 16) bias_ld(ch + 4, bw[ch & 3]);
#pragma unroll
              for (int m = 0; m < 4; ++m)
                x[4 * ch + m] = __ffma2_rn(x[4 * ch + m], sc2,
                                           make_float2(__uint_as_float(cur[m] << 16), __uint_as_float(cur[m] & 0xffff0000u)));
            }
          }
          if (mask && flags[il * C::MAXKT + kt]) {
            // the slice's mask entries of this key tile (the same for every row: broadcast loads),
            // 16 keys at a time; each chunk's address depends on the previous chunk's sums so that
            // the loads are not all hoisted next to the 128 live scores
            uint32_t maddr = smem_u32(mk + il * C::NMAX + kt * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t mw[8];
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(mw[0]), "=r"(mw[1]), "=r"(mw[2]), "=r"(mw[3])
                           : "r"(maddr));
              asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(mw[4]), "=r"(mw[5]), "=r"(mw[6]), "=r"(mw[7])
                           : "r"(maddr + 16));
#pragma unroll
              for (int m = 0; m < 8; ++m)
                x[8 * c + m] = __fadd2_rn(x[8 * c + m], make_float2(__uint_as_float(mw[m] << 16),
                                                                    __uint_as_float(mw[m] & 0xffff0000u)));
              maddr += 32;
              asm volatile("" : "+r"(maddr) : "f"(x[8 * c + 7].y));
            }
          }
          if (nvalid < 128) {
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              if (2 * e >= nvalid) x[e].x = -INFINITY;
              if (2 * e + 1 >= nvalid) x[e].y = -INFINITY;
            }
          }
          float mt;
          {  // row max with three-input max: one instruction per key pair
            float m8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) m8[c] = fmaxf(x[c].x, x[c].y);
#pragma unroll
            for (int e = 8; e < 64; ++e) m8[e & 7] = fmax3(m8[e & 7], x[e].x, x[e].y);
            mt = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
          }
          // lazy online-softmax rescale
          float alpha = 1.f;
          bool resc = false;
          float mr = m_ref[0];
#pragma unroll
          for (int qq = 1; qq < NL; ++qq)
            if (qq == sl) mr = m_ref[qq];
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
            // O_il may be touched once the P.V of this slice's key tile kt-1 has completed
            int pv = pvc[0];
#pragma unroll
            for (int qq = 1; qq < NL; ++qq)
              if (qq == sl) pv = pvc[qq];
            ok = wait_bar_warp(bar(C::B_PVDONE + il), (pv + kt - 1) & 1, ab);
            if (!ok) break;
            const uint32_t oaddr = tbase + lane_base + C::TO + il * HD;
#pragma unroll 1
            for (int c = 0; c < HD; c += 8) {  // 8 columns at a time: few registers next to the live scores
              uint32_t r[8];
              tmem_ld8(oaddr + c, r);
              tmem_wait_ld(r);
#pragma unroll
              for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st8(oaddr + c, r);
            }
          }
          const float mu = (mr == -INFINITY) ? 0.f : mr * kLog2e;
          const float2 mu2 = make_float2(-mu, -mu);
          float2 ls2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {  // keys 64*hh + [0,64): P (FP16 pairs) over S columns 64*hh + [0,32)
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float2 a = __ffma2_rn(x[32 * hh + e], l2e2, mu2);  // (x - m) in log2 units
              const float2 pv = make_float2(ex2(a.x), ex2(a.y));
              ls2[e & 3] = __fadd2_rn(ls2[e & 3], pv);
              pk[e] = pack_f16x2(pv.x, pv.y);
            }
            tmem_st32(scol + 64 * hh, pk);
          }
          const float2 lsa = __fadd2_rn(__fadd2_rn(ls2[0], ls2[1]), __fadd2_rn(ls2[2], ls2[3]));
          const float ls = lsa.x + lsa.y;
#pragma unroll
          for (int qq = 0; qq < NL; ++qq)
            if (qq == sl) {
              m_ref[qq] = mr;
              l_sum[qq] = l_sum[qq] * alpha + ls;
            }
          {
            // the tile's V, BF16 -> FP16 in place (V landed with K, before S), a share per thread
            const int st = tg % C::NST;
            float vs = vsc[0];
#pragma unroll
            for (int qq = 1; qq < NL; ++qq)
              if (qq == sl) vs = vsc[qq];
            const float2 vs2 = make_float2(vs, vs);
            ok = wait_bar(bar(C::B_KVFULL + st), (tg / C::NST) & 1, ab);
            uint4 *v = reinterpret_cast<uint4 *>(sm + C::OFF_V + st * C::TILE);
#pragma unroll
            for (int e = wtid; e < C::TILE / 16; e += 128) {
              uint4 xv = v[e];
              xv.x = bf16x2_to_f16x2_scaled2(xv.x, vs2);
              xv.y = bf16x2_to_f16x2_scaled2(xv.y, vs2);
              xv.z = bf16x2_to_f16x2_scaled2(xv.z, vs2);
              xv.w = bf16x2_to_f16x2_scaled2(xv.w, vs2);
              v[e] = xv;
            }
            fence_proxy_async_smem();
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::B_PFULL + sbuf));
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (tma_bias) {  // this thread is done with the key tile's bias
          fence_proxy_async_smem();  // order the generic-proxy reads before the TMA overwrite
          mbar_arrive(bar(C::B_BFREE + (kb & 1)));
        }
      }
      if (!ok) break;
      if (mask) {
        fence_proxy_async_smem();  // (the next copy into this buffer is an async-proxy write)
        mbar_arrive(bar(C::B_MFREE + (k & 1)));
      }
      tgu += nkt * ng;
#pragma unroll
      for (int s = 0; s < NL; ++s)
        if (wg + 2 * s < ng) pvc[s] += nkt;
      // epilogue: read O of this warpgroup's slices out of TMEM and release it, then
      // O = acc / l -> BF16, residual, LSE
      ok = wait_bar_warp(bar(C::B_OFINAL + wg), k & 1, ab);
      if (!ok) break;
      tc_fence_after();
      uint32_t oacc[NL][HD] = {};
#pragma unroll
      for (int s = 0; s < NL; ++s) {
        if (wg + 2 * s < ng) {
          const uint32_t oaddr = tbase + lane_base + C::TO + (wg + 2 * s) * HD;
          if constexpr (HD == 32) {
            tmem_ld32(oaddr, oacc[s]);
          } else {
            tmem_ld16(oaddr, oacc[s]);
          }
        }
      }
      tmem_wait_ld(oacc);
      tc_fence_before();
      mbar_arrive(bar(C::B_OFREE + wg));
#pragma unroll
      for (int s = 0; s < NL; ++s) {
        const int il = wg + 2 * s;
        if (il >= ng || j >= g.N) continue;
        const int i = i0 + il;
        const float lsum = l_sum[s];
        const float inv = lsum > 0.f ? __frcp_rn(lsum) * vinv[s] : 0.f;  // 1 / l, and V's scale undone
        uint32_t ob[HD / 2], rb[HD / 2];
#pragma unroll
        for (int c = 0; c < HD / 2; ++c) {
          const float o0 = __uint_as_float(oacc[s][2 * c]) * inv, o1 = __uint_as_float(oacc[s][2 * c + 1]) * inv;
          ob[c] = pack_bf16x2(o0, o1);
          rb[c] = pack_bf16x2(o0 - __uint_as_float(ob[c] << 16), o1 - __uint_as_float(ob[c] & 0xffff0000u));
        }
        const int64_t off = pos_row(g, b, i, j, NODE) * g.H * HD + (int64_t)h * HD;
        // the row: 64 bytes (d = 32) or 32 bytes (d = 16), 32-byte stores
#pragma unroll
        for (int c = 0; c < HD / 16; ++c) {
          asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(O + off + 16 * c), "r"(ob[8 * c]),
                       "r"(ob[8 * c + 1]), "r"(ob[8 * c + 2]), "r"(ob[8 * c + 3]), "r"(ob[8 * c + 4]),
                       "r"(ob[8 * c + 5]), "r"(ob[8 * c + 6]), "r"(ob[8 * c + 7])
                       : "memory");
          if (Ores)
            asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(Ores + off + 16 * c),
                         "r"(rb[8 * c]), "r"(rb[8 * c + 1]), "r"(rb[8 * c + 2]), "r"(rb[8 * c + 3]),
                         "r"(rb[8 * c + 4]), "r"(rb[8 * c + 5]), "r"(rb[8 * c + 6]), "r"(rb[8 * c + 7])
                         : "memory");
        }
        LSE[(((int64_t)b * g.S + i) * g.H + h) * g.N + j] = lsum > 0.f ? m_ref[s] + __log2f(lsum) * kLn2 : -INFINITY;
      }
    }
    cp_async_wait_all();
  } else {
    reg_dealloc<C::REG_OTHER>();  // warp 3 only donates registers
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

template <int HD>
cudaError_t plan_fwd_t(const Dims &g, const uint16_t *Q, const uint16_t *K, const uint16_t *V, const uint16_t *bias,
                       FwdPlan *p) {
  using C = FwdCfg<HD>;
  cudaError_t e = make_rows_map(&p->mq, Q, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&p->mk, K, g, 128);
  if (e == cudaSuccess) e = make_rows_map(&p->mv, V, g, 128);
  if (e != cudaSuccess) return e;
  if ((g.N & 7) == 0) {
    e = make_bias_map(&p->mb, bias, g.N, g.B * g.H);
    if (e != cudaSuccess) return e;
  } else {
    memset(&p->mb, 0, sizeof(p->mb));  // unused: the kernel stages the bias itself
  }
  auto *kern = g.node ? fwd_kernel<HD, 1> : fwd_kernel<HD, 0>;
  int dev = 0;
  e = current_device(&dev);
  if (e != cudaSuccess) return e;
  static DeviceOnce ready[2];  // per node
  DeviceOnce &once = ready[g.node ? 1 : 0];
  if (!once.done(dev)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    // the setmaxnreg split only balances if the kernel was built with exactly REG_LAUNCH
    // registers per thread, so refuse to launch otherwise
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != (int)C::REG_LAUNCH) return cudaErrorInvalidConfiguration;
    once.mark(dev);
  }
  // persistent: one CTA per resident slot, each walking units blockIdx.x, +gridDim.x, ...
  // (both node instantiations have the same resources)
  static DeviceValue slots;
  int nslots = slots.get(dev);
  if (nslots == 0) {
    int nsm = 0, per = 0;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, C::NTHREADS, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    if (per < 1) return cudaErrorInvalidConfiguration;
    nslots = nsm * per;
    slots.set(dev, nslots);
  }
  const int nunits = g.B * ((g.S + C::GF - 1) / C::GF) * g.H * ((g.N + 127) / 128);
  p->grid = min(nunits, nslots);
  return cudaSuccess;
}

cudaError_t plan_fwd(const Dims &g, const uint16_t *Q, const uint16_t *K, const uint16_t *V, const uint16_t *bias,
                     FwdPlan *p) {
  return g.d == 32 ? plan_fwd_t<32>(g, Q, K, V, bias, p) : plan_fwd_t<16>(g, Q, K, V, bias, p);
}

// The V scale pre-pass; it must precede launch_fwd on the same stream.
cudaError_t launch_fwd_vscale(const Dims &g, const uint16_t *V, float *LSE, cudaStream_t stream) {
  const dim3 grid(g.H, g.B * g.S);
  const uint4 *v = reinterpret_cast<const uint4 *>(V);
  int *slots = reinterpret_cast<int *>(LSE);
  if (g.d == 32) {
    if (g.node) fwd_vscale_kernel<32, 1><<<grid, 256, 0, stream>>>(g, v, slots);
    else fwd_vscale_kernel<32, 0><<<grid, 256, 0, stream>>>(g, v, slots);
  } else {
    if (g.node) fwd_vscale_kernel<16, 1><<<grid, 256, 0, stream>>>(g, v, slots);
    else fwd_vscale_kernel<16, 0><<<grid, 256, 0, stream>>>(g, v, slots);
  }
  return cudaGetLastError();
}

cudaError_t launch_fwd(const Dims &g, const FwdPlan &p, const uint16_t *bias, const uint16_t *mask, uint16_t *O,
                       float *LSE, uint16_t *Ores, int *status, cudaStream_t stream) {
  auto *kern = g.d == 32 ? (g.node ? fwd_kernel<32, 1> : fwd_kernel<32, 0>) : (g.node ? fwd_kernel<16, 1> : fwd_kernel<16, 0>);
  const int smem = g.d == 32 ? FwdCfg<32>::SMEM_ALLOC : FwdCfg<16>::SMEM_ALLOC;
  const int nthreads = g.d == 32 ? FwdCfg<32>::NTHREADS : FwdCfg<16>::NTHREADS;
  kern<<<p.grid, nthreads, smem, stream>>>(p.mq, p.mk, p.mv, p.mb, g, bias, mask, O, LSE, Ores, status);
  return cudaGetLastError();
}

}  // namespace triattn
