// Scalar (CUDA-core) forward and backward kernels: a plain, slow first GPU
// path used to pin the interface, layouts and determinism machinery. Each
// thread owns one query row (forward, dQ) or one key row (dK, dV, dBias) and
// walks the other axis in FP32.
#include "common.cuh"

namespace triattn {

constexpr int kSimtRows = 64;

__device__ __forceinline__ float ld_bf16(const uint16_t *p) { return bf16_to_f32(*p); }

template <int HD>
__global__ void __launch_bounds__(kSimtRows)
simt_fwd_kernel(Dims g, const uint16_t *__restrict__ Q, const uint16_t *__restrict__ K,
                const uint16_t *__restrict__ V, const uint16_t *__restrict__ bias,
                const uint16_t *__restrict__ mask, uint16_t *__restrict__ O,
                float *__restrict__ LSE, uint16_t *__restrict__ Ores) {
  __shared__ float sK[kSimtRows][HD + 1], sV[kSimtRows][HD + 1], sM[kSimtRows];
  const int bi = blockIdx.z, b = bi / g.S, i = bi % g.S, h = blockIdx.y;
  const int j = blockIdx.x * kSimtRows + threadIdx.x;
  const int HDs = g.H * HD;
  float q[HD], o[HD];
  const bool active = j < g.N;
#pragma unroll
  for (int c = 0; c < HD; ++c) {
    q[c] = active ? ld_bf16(Q + pos_row(g, b, i, j) * HDs + h * HD + c) : 0.f;
    o[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const uint16_t *brow = bias + (((int64_t)b * g.H + h) * g.N + (active ? j : 0)) * g.N;
  for (int k0 = 0; k0 < g.N; k0 += kSimtRows) {
    __syncthreads();
    for (int t = threadIdx.x; t < kSimtRows * HD; t += kSimtRows) {
      const int r = t / HD, c = t % HD, k = k0 + r;
      const bool ok = k < g.N;
      sK[r][c] = ok ? ld_bf16(K + pos_row(g, b, i, k) * HDs + h * HD + c) : 0.f;
      sV[r][c] = ok ? ld_bf16(V + pos_row(g, b, i, k) * HDs + h * HD + c) : 0.f;
    }
    {
      const int k = k0 + threadIdx.x;
      sM[threadIdx.x] = k < g.N ? (mask ? ld_bf16(mask + ((int64_t)b * g.S + i) * g.N + k) : 0.f) : -INFINITY;
    }
    __syncthreads();
    if (!active) continue;
    const int kn = min(kSimtRows, g.N - k0);
    for (int r = 0; r < kn; ++r) {
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < HD; ++c) dot = fmaf(q[c], sK[r][c], dot);
      const float s = dot * g.scale + ld_bf16(brow + k0 + r) + sM[r];
      if (s == -INFINITY) continue;
      if (s > m) {
        const float corr = (m == -INFINITY) ? 0.f : expf(m - s);
        l *= corr;
#pragma unroll
        for (int c = 0; c < HD; ++c) o[c] *= corr;
        m = s;
      }
      const float p = expf(s - m);
      l += p;
#pragma unroll
      for (int c = 0; c < HD; ++c) o[c] = fmaf(p, sV[r][c], o[c]);
    }
  }
  if (!active) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int64_t base = pos_row(g, b, i, j) * HDs + h * HD;
#pragma unroll
  for (int c = 0; c < HD; ++c) {
    const float of = o[c] * inv;
    const uint16_t ob = f32_to_bf16_rn(of);
    O[base + c] = ob;
    if (Ores) Ores[base + c] = f32_to_bf16_rn(of - bf16_to_f32(ob));
  }
  LSE[(((int64_t)b * g.S + i) * g.H + h) * g.N + j] = l > 0.f ? m + logf(l) : -INFINITY;
}

// Key-row kernel: dK, dV for every slice and the dBias partial of one slice
// group (slices [g0, g1)); the partial is accumulated in slice order by the
// thread that owns the key column, so the sum order is fixed.
template <int HD>
__global__ void __launch_bounds__(kSimtRows)
simt_bwd_kv_kernel(Dims g, int G, const uint16_t *__restrict__ Q, const uint16_t *__restrict__ K,
                   const uint16_t *__restrict__ V, const uint16_t *__restrict__ bias,
                   const uint16_t *__restrict__ mask, const float *__restrict__ LSE,
                   const float *__restrict__ Dv, const uint16_t *__restrict__ dO,
                   uint16_t *__restrict__ dK, uint16_t *__restrict__ dV, float *__restrict__ partial) {
  __shared__ float sQ[kSimtRows][HD + 1], sO[kSimtRows][HD + 1], sL[kSimtRows], sD[kSimtRows];
  const int b = blockIdx.z / G, grp = blockIdx.z % G, h = blockIdx.y;
  const int g0 = (int)((int64_t)grp * g.S / G), g1 = (int)((int64_t)(grp + 1) * g.S / G);
  const int k = blockIdx.x * kSimtRows + threadIdx.x;
  const bool active = k < g.N;
  const int HDs = g.H * HD;
  const int64_t nn = (int64_t)g.N * g.N;
  float *part = partial + ((int64_t)grp * g.B * g.H + (int64_t)b * g.H + h) * nn;
  const uint16_t *bcol = bias + ((int64_t)b * g.H + h) * nn + (active ? k : 0);
  for (int i = g0; i < g1; ++i) {
    float kk[HD], vv[HD], dk[HD], dv[HD];
#pragma unroll
    for (int c = 0; c < HD; ++c) {
      kk[c] = active ? ld_bf16(K + pos_row(g, b, i, k) * HDs + h * HD + c) : 0.f;
      vv[c] = active ? ld_bf16(V + pos_row(g, b, i, k) * HDs + h * HD + c) : 0.f;
      dk[c] = 0.f;
      dv[c] = 0.f;
    }
    const float mk = (active && mask) ? ld_bf16(mask + ((int64_t)b * g.S + i) * g.N + k) : 0.f;
    for (int j0 = 0; j0 < g.N; j0 += kSimtRows) {
      __syncthreads();
      for (int t = threadIdx.x; t < kSimtRows * HD; t += kSimtRows) {
        const int r = t / HD, c = t % HD, j = j0 + r;
        const bool ok = j < g.N;
        sQ[r][c] = ok ? ld_bf16(Q + pos_row(g, b, i, j) * HDs + h * HD + c) : 0.f;
        sO[r][c] = ok ? ld_bf16(dO + pos_row(g, b, i, j) * HDs + h * HD + c) : 0.f;
      }
      {
        const int j = j0 + threadIdx.x;
        const int64_t li = (((int64_t)b * g.S + i) * g.H + h) * g.N + j;
        sL[threadIdx.x] = j < g.N ? LSE[li] : -INFINITY;
        sD[threadIdx.x] = j < g.N ? Dv[li] : 0.f;
      }
      __syncthreads();
      if (!active) continue;
      const int jn = min(kSimtRows, g.N - j0);
      for (int r = 0; r < jn; ++r) {
        const int j = j0 + r;
        float dot = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < HD; ++c) {
          dot = fmaf(sQ[r][c], kk[c], dot);
          dp = fmaf(sO[r][c], vv[c], dp);
        }
        const float s = dot * g.scale + ld_bf16(bcol + (int64_t)j * g.N) + mk;
        const float p = (sL[r] == -INFINITY || s == -INFINITY) ? 0.f : expf(s - sL[r]);
        const float ds = p * (dp - sD[r]);
#pragma unroll
        for (int c = 0; c < HD; ++c) {
          dv[c] = fmaf(p, sO[r][c], dv[c]);
          dk[c] = fmaf(ds, sQ[r][c], dk[c]);
        }
        float *pp = part + (int64_t)j * g.N + k;
        *pp = (i == g0) ? ds : (*pp + ds);
      }
    }
    if (active) {
      const int64_t base = pos_row(g, b, i, k) * HDs + h * HD;
#pragma unroll
      for (int c = 0; c < HD; ++c) {
        dK[base + c] = f32_to_bf16_rn(dk[c] * g.scale);
        dV[base + c] = f32_to_bf16_rn(dv[c]);
      }
    }
  }
}

template <int HD>
__global__ void __launch_bounds__(kSimtRows)
simt_bwd_q_kernel(Dims g, const uint16_t *__restrict__ Q, const uint16_t *__restrict__ K,
                  const uint16_t *__restrict__ V, const uint16_t *__restrict__ bias,
                  const uint16_t *__restrict__ mask, const float *__restrict__ LSE,
                  const float *__restrict__ Dv, const uint16_t *__restrict__ dO,
                  uint16_t *__restrict__ dQ) {
  __shared__ float sK[kSimtRows][HD + 1], sV[kSimtRows][HD + 1], sM[kSimtRows];
  const int bi = blockIdx.z, b = bi / g.S, i = bi % g.S, h = blockIdx.y;
  const int j = blockIdx.x * kSimtRows + threadIdx.x;
  const bool active = j < g.N;
  const int HDs = g.H * HD;
  float q[HD], o[HD], dq[HD];
#pragma unroll
  for (int c = 0; c < HD; ++c) {
    q[c] = active ? ld_bf16(Q + pos_row(g, b, i, j) * HDs + h * HD + c) : 0.f;
    o[c] = active ? ld_bf16(dO + pos_row(g, b, i, j) * HDs + h * HD + c) : 0.f;
    dq[c] = 0.f;
  }
  const int64_t li = (((int64_t)b * g.S + i) * g.H + h) * g.N + (active ? j : 0);
  const float lse = LSE[li], Dj = Dv[li];
  const uint16_t *brow = bias + (((int64_t)b * g.H + h) * g.N + (active ? j : 0)) * g.N;
  for (int k0 = 0; k0 < g.N; k0 += kSimtRows) {
    __syncthreads();
    for (int t = threadIdx.x; t < kSimtRows * HD; t += kSimtRows) {
      const int r = t / HD, c = t % HD, k = k0 + r;
      const bool ok = k < g.N;
      sK[r][c] = ok ? ld_bf16(K + pos_row(g, b, i, k) * HDs + h * HD + c) : 0.f;
      sV[r][c] = ok ? ld_bf16(V + pos_row(g, b, i, k) * HDs + h * HD + c) : 0.f;
    }
    {
      const int k = k0 + threadIdx.x;
      sM[threadIdx.x] = k < g.N ? (mask ? ld_bf16(mask + ((int64_t)b * g.S + i) * g.N + k) : 0.f) : -INFINITY;
    }
    __syncthreads();
    if (!active) continue;
    const int kn = min(kSimtRows, g.N - k0);
    for (int r = 0; r < kn; ++r) {
      float dot = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < HD; ++c) {
        dot = fmaf(q[c], sK[r][c], dot);
        dp = fmaf(o[c], sV[r][c], dp);
      }
      const float s = dot * g.scale + ld_bf16(brow + k0 + r) + sM[r];
      const float p = (lse == -INFINITY || s == -INFINITY) ? 0.f : expf(s - lse);
      const float ds = p * (dp - Dj);
#pragma unroll
      for (int c = 0; c < HD; ++c) dq[c] = fmaf(ds, sK[r][c], dq[c]);
    }
  }
  if (!active) return;
  const int64_t base = pos_row(g, b, i, j) * HDs + h * HD;
#pragma unroll
  for (int c = 0; c < HD; ++c) dQ[base + c] = f32_to_bf16_rn(dq[c] * g.scale);
}

cudaError_t launch_simt_fwd(const Dims &g, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                            const uint16_t *bias, const uint16_t *mask, uint16_t *O, float *LSE,
                            uint16_t *Ores, cudaStream_t stream) {
  dim3 grid((g.N + kSimtRows - 1) / kSimtRows, g.H, g.B * g.S);
  if (g.d == 32)
    simt_fwd_kernel<32><<<grid, kSimtRows, 0, stream>>>(g, Q, K, V, bias, mask, O, LSE, Ores);
  else
    simt_fwd_kernel<16><<<grid, kSimtRows, 0, stream>>>(g, Q, K, V, bias, mask, O, LSE, Ores);
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd(const Dims &g, int G, const uint16_t *Q, const uint16_t *K,
                            const uint16_t *V, const uint16_t *bias, const uint16_t *mask,
                            const float *LSE, const float *Dv, const uint16_t *dO, uint16_t *dQ,
                            uint16_t *dK, uint16_t *dV, float *partial, cudaStream_t stream) {
  dim3 gkv((g.N + kSimtRows - 1) / kSimtRows, g.H, g.B * G);
  dim3 gq((g.N + kSimtRows - 1) / kSimtRows, g.H, g.B * g.S);
  if (g.d == 32) {
    simt_bwd_kv_kernel<32><<<gkv, kSimtRows, 0, stream>>>(g, G, Q, K, V, bias, mask, LSE, Dv, dO, dK, dV, partial);
    simt_bwd_q_kernel<32><<<gq, kSimtRows, 0, stream>>>(g, Q, K, V, bias, mask, LSE, Dv, dO, dQ);
  } else {
    simt_bwd_kv_kernel<16><<<gkv, kSimtRows, 0, stream>>>(g, G, Q, K, V, bias, mask, LSE, Dv, dO, dK, dV, partial);
    simt_bwd_q_kernel<16><<<gq, kSimtRows, 0, stream>>>(g, Q, K, V, bias, mask, LSE, Dv, dO, dQ);
  }
  return cudaGetLastError();
}

}  // namespace triattn
