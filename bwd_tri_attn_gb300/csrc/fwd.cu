// Forward pass: tcgen05/TMEM flash-style kernel with the pair bias staged in
// shared memory and reused across the slices of a CTA.
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract): each row-slice of the pair
// tensor runs attention with a pair bias shared by all slices; the forward
// keeps BF16 outputs and, for the backward correction, a BF16 approximation of
// the output-rounding residual (O_fp32 - bf16(O)), without changing O.
//
// Work unit (one CTA): batch b, head h, query tile jt (128 rows), and a group
// of GF consecutive slices. For every key tile kt the bias tile
// bias[b,h,jt,kt] is brought into shared memory once (each softmax thread
// stages and converts its own query row) and used for all GF slices:
//   S_i  = Q_i K_i^T           tcgen05 (BF16 x BF16 -> FP32 TMEM), M=128, N=128
//   P_i  = exp2(S_i*scale*log2e + bias*log2e - m_i)   online softmax, FP32
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
// O is rescaled in TMEM only then.
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
  static constexpr int OFF_BF = OFF_V + NST * TILE;         // FP32 bias*log2e rows: 128 x 512 B
  static constexpr int OFF_BS = OFF_BF + 128 * 512;         // BF16 bias staging rows: 128 x 256 B
  static constexpr int OFF_MASK = OFF_BS + 128 * 256;       // FP32 mask*log2e [GF][NMAX]
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
  static constexpr int NBAR = B_OFINAL + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int NSOFT = 8, WARP_TMA = 8, WARP_MMA = 9, WARP_CV = 10, NTHREADS = 352;
  static constexpr uint32_t TO = NSB * 128;  // O accumulators: TO + i*d
  static_assert(TO + GF * HD <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

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
  const int jt = blockIdx.x, h = blockIdx.y;
  const int ngroups = (g.S + C::GF - 1) / C::GF;
  const int b = blockIdx.z / ngroups, i0 = (blockIdx.z % ngroups) * C::GF;
  const int ng = min(C::GF, g.S - i0);
  const int nkt = (g.N + 127) / 128;
  const int T = nkt * ng;
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
    int issued = 0;
    if (lane == 0) {
      tma_prefetch_map(&mQ);
      tma_prefetch_map(&mK);
      tma_prefetch_map(&mV);
      mbar_arrive_expect_tx(bar(C::B_Q), ng * C::TILE);
      for (int il = 0; il < ng; ++il)
        tma_load_4d(sb0 + C::OFF_Q + il * C::TILE, &mQ, bar(C::B_Q), 0, h, jt * 128, b * g.S + i0 + il);
    }
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int st = t % C::NST, use = t / C::NST;
      if (use > 0) ok = wait_bar_warp(bar(C::B_KVEMPTY + st), (use - 1) & 1, ab);
      if (!ok) break;
      if (lane == 0) {
        const int kt = t / ng, il = t % ng;
        mbar_arrive_expect_tx(bar(C::B_KVFULL + st), 2 * C::TILE);
        tma_load_4d(sb0 + C::OFF_K + st * C::TILE, &mK, bar(C::B_KVFULL + st), 0, h, kt * 128, b * g.S + i0 + il);
        tma_load_4d(sb0 + C::OFF_V + st * C::TILE, &mV, bar(C::B_KVFULL + st), 0, h, kt * 128, b * g.S + i0 + il);
      }
      issued = t + 1;
    }
    if (!ok && lane == 0) {
      // drain loads still in flight before the CTA's shared memory goes away
      drain_bar(bar(C::B_Q), 0);
      for (int t = max(0, issued - C::NST); t < issued; ++t) drain_bar(bar(C::B_KVFULL + t % C::NST), (t / C::NST) & 1);
    }
  } else if (warp == C::WARP_CV) {
    // ------------------------------------------------------------ V: BF16 -> FP16 in shared memory
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int st = t % C::NST, use = t / C::NST;
      ok = wait_bar_warp(bar(C::B_KVFULL + st), use & 1, ab);
      if (!ok) break;
      uint4 *v = reinterpret_cast<uint4 *>(sm + C::OFF_V + st * C::TILE);
      for (int e = lane; e < C::TILE / 16; e += 32) {
        uint4 w = v[e];
        w.x = bf16x2_to_f16x2(w.x);
        w.y = bf16x2_to_f16x2(w.y);
        w.z = bf16x2_to_f16x2(w.z);
        w.w = bf16x2_to_f16x2(w.w);
        v[e] = w;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_VREADY + st));
    }
  } else if (warp == C::WARP_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(128, 128, true, true, false, false);
      constexpr uint32_t idPV = idesc_f16(128, HD, false, false, false, true);
      auto issue_pv = [&](int t) -> bool {
        const int kt = t / ng, il = t % ng, sbuf = t % C::NSB, st = t % C::NST;
        if (!wait_bar(bar(C::B_PFULL + sbuf), (t / C::NSB) & 1, ab)) return false;
        if (!wait_bar(bar(C::B_VREADY + st), (t / C::NST) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t vaddr = sb0 + C::OFF_V + st * C::TILE;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tbase + C::TO + il * HD, tbase + sbuf * 128 + (ks >> 2) * 64 + (ks & 3) * 8,
                 smem_desc(vaddr + ks * 16 * C::ROWB, 16, 8 * C::ROWB, C::SW), idPV, (kt > 0 || ks > 0) ? 1u : 0u);
        mma_commit(bar(C::B_SFREE + sbuf));
        mma_commit(bar(C::B_KVEMPTY + st));
        mma_commit(bar(C::B_PVDONE + il));
        return true;
      };
      bool ok = wait_bar(bar(C::B_Q), 0, ab);
      for (int t = 0; t < T && ok; ++t) {
        const int st = t % C::NST, sbuf = t % C::NSB, il = t % ng;
        ok = wait_bar(bar(C::B_KVFULL + st), (t / C::NST) & 1, ab);
        if (ok && t >= C::NSB) ok = wait_bar(bar(C::B_SFREE + sbuf), ((t / C::NSB) - 1) & 1, ab);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qaddr = sb0 + C::OFF_Q + il * C::TILE, kaddr = sb0 + C::OFF_K + st * C::TILE;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks)
          mma_ss(tbase + sbuf * 128, smem_desc(qaddr + ks * 32, 16, 8 * C::ROWB, C::SW),
                 smem_desc(kaddr + ks * 32, 16, 8 * C::ROWB, C::SW), idS, ks > 0 ? 1u : 0u);
        mma_commit(bar(C::B_SFULL + sbuf));
        if (t >= 1) ok = issue_pv(t - 1);
      }
      if (ok) ok = issue_pv(T - 1);
      mma_commit(bar(C::B_OFINAL));
      drain_bar(bar(C::B_OFINAL), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue (warps 0-7)
    // Two threads per query row: warp w handles TMEM lane quarter q = w % 4 and
    // the key half w / 4 (64 of the tile's 128 keys).
    const int q = warp & 3, half = warp >> 2;
    const int row = q * 32 + lane;
    const int j = jt * 128 + row;
    const int jr = min(j, g.N - 1);  // rows past N reuse a valid bias row; their outputs are dropped
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t pair_bar = 2 + q;  // named barrier of the two warps sharing these rows
    float *maskf = reinterpret_cast<float *>(sm + C::OFF_MASK);
    int *flags = reinterpret_cast<int *>(sm + C::OFF_FLAG);
    float *xmax = reinterpret_cast<float *>(sm + C::OFF_XCH);  // [2 parities][2 halves][128 rows]
    const float c1 = g.scale * kLog2e;
    const float2 c1x2 = make_float2(c1, c1);

    // bias row: this thread stages and converts its half (64 keys) of row jr for every key tile
    const uint16_t *brow = bias + (((int64_t)b * g.H + h) * g.N + jr) * g.N;
    const uint32_t stage_row = sb0 + C::OFF_BS + row * 256;
    const uint32_t bf_row = sb0 + C::OFF_BF + row * 512;
    const uint32_t sw = row & 7;
    auto stage_bias = [&](int kt) {
      const int k0 = kt * 128 + half * 64, nv = min(64, g.N - k0);
      const uint16_t *src = brow + k0;
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
    auto convert_bias = [&](int kt) {
      const int nv = min(64, g.N - kt * 128 - half * 64);
#pragma unroll 2
      for (int cl = 0; cl < 8; ++cl) {
        const int c = half * 8 + cl;
        uint32_t w[4];
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "r"(stage_row + ((c ^ sw) << 4)));
        float f[8];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          f[2 * qq] = __uint_as_float(w[qq] << 16) * kLog2e;
          f[2 * qq + 1] = __uint_as_float(w[qq] & 0xffff0000u) * kLog2e;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (cl * 8 + e >= nv) f[e] = -INFINITY;
        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(bf_row + (((2 * c) ^ sw) << 4)), "f"(f[0]),
                     "f"(f[1]), "f"(f[2]), "f"(f[3])
                     : "memory");
        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(bf_row + (((2 * c + 1) ^ sw) << 4)),
                     "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
                     : "memory");
      }
    };

    stage_bias(0);  // first bias tile in flight while the mask rows load
    // per-slice additive mask (log2 units) and per-tile "has a nonzero entry" flags
    if (tid < C::GF * C::MAXKT) flags[tid] = 0;
    named_sync(1, 256);
    if (mask) {
      for (int il0 = 0; il0 < ng; il0 += 2) {  // two slices per memory round trip
        float v[2][C::NMAX / 256];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int m = 0; m < C::NMAX / 256; ++m) {
            const int il = il0 + a, k = tid + 256 * m;
            v[a][m] = (il < ng && k < g.N) ? bf16_to_f32(mask[((int64_t)b * g.S + i0 + il) * g.N + k]) * kLog2e : 0.f;
          }
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int m = 0; m < C::NMAX / 256; ++m) {
            const int il = il0 + a, k = tid + 256 * m;
            if (il < ng && k < nkt * 128) {
              maskf[il * C::NMAX + k] = v[a][m];
              if (v[a][m] != 0.f) flags[il * C::MAXKT + (k >> 7)] = 1;  // every writer stores the same value
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
    bool ok = true;
    for (int kt = 0; kt < nkt && ok; ++kt) {
      cp_async_wait_all();
      convert_bias(kt);
      if (kt + 1 < nkt) stage_bias(kt + 1);
#pragma unroll 1
      for (int il = 0; il < ng; ++il) {
        const int t = kt * ng + il, sbuf = t % C::NSB;
        ok = wait_bar_warp(bar(C::B_SFULL + sbuf), (t / C::NSB) & 1, ab);
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
        // scores in log2 units: S*scale*log2e + bias*log2e (+ mask*log2e)
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          float4 bv;
          asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                       : "=f"(bv.x), "=f"(bv.y), "=f"(bv.z), "=f"(bv.w)
                       : "r"(bf_row + (((half * 16 + ch) ^ sw) << 4)));
          x[2 * ch] = __ffma2_rn(x[2 * ch], c1x2, make_float2(bv.x, bv.y));
          x[2 * ch + 1] = __ffma2_rn(x[2 * ch + 1], c1x2, make_float2(bv.z, bv.w));
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
        xmax[((t & 1) * 2 + half) * 128 + row] = mloc;
        named_sync(pair_bar, 64);
        const float mt = fmaxf(mloc, xmax[((t & 1) * 2 + (half ^ 1)) * 128 + row]);
        // lazy online-softmax rescale (the same decision in both threads of the row)
        float alpha = 1.f;
        bool resc = false;
        float mr = m_ref[0];
#pragma unroll
        for (int qq = 1; qq < C::GF; ++qq)
          if (qq == il) mr = m_ref[qq];
        if (kt == 0) {
          mr = mt;
        } else if (mt > mr + 8.f) {
          if (mr == -INFINITY) {
            mr = mt;  // O_i and l_i are still exactly zero
          } else {
            alpha = ex2(mr - mt);
            resc = true;
            mr = mt;
          }
        }
        if (__any_sync(0xffffffffu, resc)) {
          ok = wait_bar_warp(bar(C::B_PVDONE + il), (kt - 1) & 1, ab);
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
        const float mu = (mr == -INFINITY) ? 0.f : mr;
        const float2 mu2 = make_float2(-mu, -mu);
        float2 ls2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 a = __fadd2_rn(x[e], mu2);
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
    // epilogue: O = acc / l -> BF16, residual, LSE
    if (ok) ok = wait_bar_warp(bar(C::B_OFINAL), 0, ab);
    if (ok) {
      tc_fence_after();
      float *xl = reinterpret_cast<float *>(sm + C::OFF_XCH) + 4 * 128;  // [GF][2 halves][128 rows]
#pragma unroll
      for (int qq = 0; qq < C::GF; ++qq) xl[(qq * 2 + half) * 128 + row] = l_sum[qq];
      named_sync(pair_bar, 64);
#pragma unroll 1
      for (int il = 0; il < ng; ++il) {
        const float lsum = xl[(il * 2 + 0) * 128 + row] + xl[(il * 2 + 1) * 128 + row];
        float mref = -INFINITY;
#pragma unroll
        for (int qq = 0; qq < C::GF; ++qq)
          if (qq == il) mref = m_ref[qq];
        uint32_t r[HD / 2];
        const uint32_t oaddr = tbase + lane_base + C::TO + il * HD + half * (HD / 2);
        if constexpr (HD == 32) {
          tmem_ld16(oaddr, r);
        } else {
          tmem_ld8(oaddr, r);
        }
        tmem_wait_ld(r);
        if (j < g.N) {
          const int i = i0 + il;
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
          uint32_t ob[HD / 4], rb[HD / 4];
#pragma unroll
          for (int c = 0; c < HD / 4; ++c) {
            const float o0 = __uint_as_float(r[2 * c]) * inv, o1 = __uint_as_float(r[2 * c + 1]) * inv;
            const uint16_t a0 = f32_to_bf16_rn(o0), a1 = f32_to_bf16_rn(o1);
            ob[c] = (uint32_t)a0 | ((uint32_t)a1 << 16);
            rb[c] = (uint32_t)f32_to_bf16_rn(o0 - bf16_to_f32(a0)) |
                    ((uint32_t)f32_to_bf16_rn(o1 - bf16_to_f32(a1)) << 16);
          }
          const int64_t off = pos_row(g, b, i, j) * g.H * HD + (int64_t)h * HD + half * (HD / 2);
          uint4 *od = reinterpret_cast<uint4 *>(O + off);
#pragma unroll
          for (int c = 0; c < HD / 16; ++c) od[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
          if (Ores) {
            uint4 *rd = reinterpret_cast<uint4 *>(Ores + off);
#pragma unroll
            for (int c = 0; c < HD / 16; ++c)
              rd[c] = make_uint4(rb[4 * c], rb[4 * c + 1], rb[4 * c + 2], rb[4 * c + 3]);
          }
          if (half == 0)
            LSE[(((int64_t)b * g.S + i) * g.H + h) * g.N + j] =
                lsum > 0.f ? (mref + __log2f(lsum)) * kLn2 : -INFINITY;
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
  const int ngroups = (g.S + C::GF - 1) / C::GF;
  dim3 grid((g.N + 127) / 128, g.H, g.B * ngroups);
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
