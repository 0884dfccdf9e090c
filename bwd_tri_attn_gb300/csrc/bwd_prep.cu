// Backward preparation (HBM-bound streaming kernel): the softmax-backward correction D and the
// operand scale exponents of every (batch, slice, head).
//
// D[b,i,h,j] = sum_c dO[b,i,j,h,c] * (O[b,i,j,h,c] + Ores[b,i,j,h,c]) in FP32.
//
// TurboPairFormer (arXiv 2610.05854v1, Abstract): computing this correction
// from the BF16-rounded forward output loses precision; adding back the
// stored BF16 approximation of the output-rounding residual recovers the FP32
// output to within BF16-of-a-residual, so D is formed in FP32 from O + Ores.
// With Ores == NULL the kernel uses O alone (the uncompensated variant).
//
// Scale exponents: for the main backward's FP16 operands, the largest BF16 exponent field of each
// (b, h) block of Q, K, V and dO (over all slices and positions) is accumulated with an integer
// atomicMax (order-free) into an int4 per (b, h) that the bias transpose kernel zeroed; the main
// kernel derives its power-of-two scales from it (common.cuh).
//
// Work split: one CTA per (b, i, h) and chunk of kPrepPos positions, heads fastest so that the
// CTAs running at once read whole pair-tensor rows between them (small CTAs: many waves, a short
// tail). Each thread loads one 16-byte chunk (8 BF16) of each tensor per
// position; the d/8 chunks of one position sit in neighbouring lanes and are combined with a fixed
// xor-shuffle tree, so the summation order is fixed. The exponent maxima are order-free.
#include "common.cuh"
#include "plan.cuh"

namespace triattn {

constexpr int kPrepThreads = 256;
constexpr int kPrepPos = 256;  // positions per CTA

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

template <int HD, bool kResidual, int NODE>
__global__ void __launch_bounds__(kPrepThreads)
bwd_prep_kernel(Dims g, const uint4 *__restrict__ dO, const uint4 *__restrict__ O, const uint4 *__restrict__ Ores,
                const uint4 *__restrict__ Q, const uint4 *__restrict__ K, const uint4 *__restrict__ V,
                float *__restrict__ Dout, int *__restrict__ emax) {
  __shared__ int red[kPrepThreads / 32];
  constexpr int CPH = HD / 8;               // 16-byte chunks per (position, head)
  constexpr int PPP = kPrepThreads / CPH;   // positions per pass
  const int h = blockIdx.x;
  const int bi = blockIdx.y;  // b * S + i
  const int jbeg = blockIdx.z * kPrepPos, jend = min(g.N, jbeg + kPrepPos);
  const int b = bi / g.S, i = bi - b * g.S;
  const int c = threadIdx.x % CPH, pl = threadIdx.x / CPH;
  const int cpp = g.H * CPH;  // chunks per position row
  uint32_t mq = 0, mk = 0, mv = 0, mo = 0;
  float *drow = Dout + ((int64_t)bi * g.H + h) * g.N;
  for (int j0 = jbeg; j0 < jend; j0 += PPP) {  // every lane runs every pass: the shuffle stays converged
    const int j = j0 + pl;
    float acc = 0.f;
    if (j < jend) {
      const int64_t idx = pos_row(g, b, i, j, NODE) * cpp + h * CPH + c;
      const uint4 a = ld_stream(dO + idx), o = ld_stream(O + idx);
      const uint4 q = ld_stream(Q + idx), k = ld_stream(K + idx), v = ld_stream(V + idx);
      uint4 r = make_uint4(0u, 0u, 0u, 0u);
      if (kResidual) r = ld_stream(Ores + idx);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, ov[4] = {o.x, o.y, o.z, o.w}, rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = bf2_to_f2(av[e]), fo = bf2_to_f2(ov[e]);
        if (kResidual) {
          const float2 fr = bf2_to_f2(rv[e]);
          acc = fmaf(fa.x, fo.x + fr.x, acc);
          acc = fmaf(fa.y, fo.y + fr.y, acc);
        } else {
          acc = fmaf(fa.x, fo.x, acc);
          acc = fmaf(fa.y, fo.y, acc);
        }
      }
      mo = exp_max4(mo, a);
      mq = exp_max4(mq, q);
      mk = exp_max4(mk, k);
      mv = exp_max4(mv, v);
    }
#pragma unroll
    for (int off = 1; off < CPH; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (c == 0 && j < jend) drow[j] = acc;
  }
  const int eq = block_max<kPrepThreads>(bf16x2_exp_final(mq), red);
  const int ek = block_max<kPrepThreads>(bf16x2_exp_final(mk), red);
  const int ev = block_max<kPrepThreads>(bf16x2_exp_final(mv), red);
  const int eo = block_max<kPrepThreads>(bf16x2_exp_final(mo), red);
  if (threadIdx.x < 4) {
    const int e = threadIdx.x == 0 ? eq : threadIdx.x == 1 ? ek : threadIdx.x == 2 ? ev : eo;
    if (e) atomicMax(emax + 4 * ((int64_t)b * g.H + h) + threadIdx.x, e);
  }
}

template <int HD, bool kResidual>
static cudaError_t launch_prep_t(const Dims &g, const uint4 *a, const uint4 *o, const uint4 *r, const uint4 *q,
                                 const uint4 *k, const uint4 *v, float *Dout, int *emax, cudaStream_t stream) {
  const dim3 grid(g.H, g.B * g.S, (g.N + kPrepPos - 1) / kPrepPos);
  if (g.node)
    bwd_prep_kernel<HD, kResidual, 1><<<grid, kPrepThreads, 0, stream>>>(g, a, o, r, q, k, v, Dout, emax);
  else
    bwd_prep_kernel<HD, kResidual, 0><<<grid, kPrepThreads, 0, stream>>>(g, a, o, r, q, k, v, Dout, emax);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const Dims &g, const uint16_t *dO, const uint16_t *O, const uint16_t *Ores,
                            const uint16_t *Q, const uint16_t *K, const uint16_t *V, float *Dout, int *emax,
                            cudaStream_t stream) {
  auto u = [](const uint16_t *p) { return reinterpret_cast<const uint4 *>(p); };
  if (g.d == 32) {
    if (Ores) return launch_prep_t<32, true>(g, u(dO), u(O), u(Ores), u(Q), u(K), u(V), Dout, emax, stream);
    return launch_prep_t<32, false>(g, u(dO), u(O), nullptr, u(Q), u(K), u(V), Dout, emax, stream);
  }
  if (Ores) return launch_prep_t<16, true>(g, u(dO), u(O), u(Ores), u(Q), u(K), u(V), Dout, emax, stream);
  return launch_prep_t<16, false>(g, u(dO), u(O), nullptr, u(Q), u(K), u(V), Dout, emax, stream);
}

}  // namespace triattn
