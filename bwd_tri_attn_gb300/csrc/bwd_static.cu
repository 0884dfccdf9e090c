// tri_attn_bwd_static: the backward pass with its scratch taken from a
// file-scope device array instead of a caller-provided workspace, for callers
// that cannot allocate device memory at call time (see include/tri_attn.h).
#include <math.h>
#include <mutex>

#include "common.cuh"

#include "plan.cuh"

using namespace triattn;

// The scratch array. In host code this name is only a stand-in for the symbol:
// its device address comes from cudaGetSymbolAddress (static_scratch below).
static __device__ __align__(256) unsigned char g_static_scratch[TRI_ATTN_STATIC_WORKSPACE_BYTES];

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device, looked up once per device.
unsigned char *static_scratch() {
  static std::mutex mu;
  static unsigned char *addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned char *>(p);
  }
  return addr[dev];
}

}  // namespace

namespace triattn {

// Scratch layout of tri_attn_bwd_static inside the static array: D [B,S,H,N] FP32 | exponent
// maxima [B,H][4] int | transposed bias [B*H][NP][NP] BF16 | dBias partials
// [B*H][slots][NP][NP] FP32.
struct StaticLayout {
  size_t scl_off, biast_off, partial_off, one_partial;
};

static StaticLayout static_layout(const tri_attn_shape &s) {
  const size_t NP = (size_t)(s.N + 127) / 128 * 128;
  StaticLayout l;
  l.scl_off = align_up(sizeof(float) * (size_t)s.B * s.S * s.H * s.N);
  l.biast_off = l.scl_off + align_up(16 * (size_t)s.B * s.H);
  l.partial_off = l.biast_off + align_up(2 * (size_t)s.B * s.H * NP * NP);
  l.one_partial = sizeof(float) * (size_t)s.B * s.H * NP * NP;
  return l;
}

static int check_static_args(const tri_attn_shape &s) {
  if (s.B < 1 || s.S < 1 || s.N < 1 || s.H < 1 || !isfinite(s.scale)) return TRI_ATTN_ERR_INVALID_ARG;
  if (s.node != TRI_ATTN_NODE_STARTING && s.node != TRI_ATTN_NODE_ENDING) return TRI_ATTN_ERR_INVALID_ARG;
  if ((s.d != 16 && s.d != 32) || s.N > TRI_ATTN_MAX_N || s.H > TRI_ATTN_MAX_H) return TRI_ATTN_ERR_UNSUPPORTED;
  if ((int64_t)s.B * s.S > 65535 || (int64_t)s.B * s.H * s.S > (1ll << 30)) return TRI_ATTN_ERR_UNSUPPORTED;
  return TRI_ATTN_OK;
}

// The split tri_attn_bwd_static uses: the device's split, with fewer clusters while a head would
// need more dBias partial slots than the array holds next to the other scratch.
int static_bwd_split(const tri_attn_shape &s, BwdSplit *sp) {
  int rc = check_static_args(s);
  if (rc) return rc;
  const StaticLayout l = static_layout(s);
  const size_t cap = TRI_ATTN_STATIC_WORKSPACE_BYTES;
  if (l.partial_off + l.one_partial > cap) return TRI_ATTN_ERR_STATIC_TOO_SMALL;
  const size_t fit = (cap - l.partial_off) / l.one_partial;  // partial slots per head that fit
  const Dims g{s.B, s.S, s.N, s.H, s.d, s.scale, s.node};
  if (bwd_split_active(g, sp) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  while (sp->NC > 1 && (size_t)sp->KMAX > fit) sp->KMAX = bwd_slots_for(g, --sp->NC);
  if ((size_t)sp->KMAX > fit) return TRI_ATTN_ERR_STATIC_TOO_SMALL;
  return TRI_ATTN_OK;
}

}  // namespace triattn

extern "C" int tri_attn_bwd_static(tri_attn_shape s, const tri_attn_bf16 *Q, const tri_attn_bf16 *K,
                                   const tri_attn_bf16 *V, const tri_attn_bf16 *bias, const tri_attn_bf16 *mask,
                                   const tri_attn_bf16 *O, const tri_attn_bf16 *Ores, const float *LSE,
                                   const tri_attn_bf16 *dO, tri_attn_bf16 *dQ, tri_attn_bf16 *dK, tri_attn_bf16 *dV,
                                   tri_attn_bf16 *dBias, void *stream) {
  int rc = check_static_args(s);
  if (rc) return rc;
  if (!Q || !K || !V || !bias || !O || !LSE || !dO || !dQ || !dK || !dV || !dBias) return TRI_ATTN_ERR_INVALID_ARG;
  const void *ptrs[] = {Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return TRI_ATTN_ERR_UNSUPPORTED;
  BwdSplit sp;
  rc = static_bwd_split(s, &sp);  // also refuses shapes that do not fit, before anything is enqueued
  if (rc) return rc;
  const StaticLayout l = static_layout(s);
  const Dims g{s.B, s.S, s.N, s.H, s.d, s.scale, s.node};
  unsigned char *ws = static_scratch();
  int *status = device_status_word();
  if (!ws || !status) return TRI_ATTN_ERR_CUDA;
  float *Dv = reinterpret_cast<float *>(ws);
  int *emax = reinterpret_cast<int *>(ws + l.scl_off);
  uint16_t *biasT = reinterpret_cast<uint16_t *>(ws + l.biast_off);
  float *partial = reinterpret_cast<float *>(ws + l.partial_off);
  auto st = static_cast<cudaStream_t>(stream);
  BwdPlan plan;
  if (plan_bwd(g, sp, Q, K, V, dO, biasT, dK, dV, &plan) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  cudaError_t e = launch_bias_transpose(g, bias, biasT, emax, st);
  if (e == cudaSuccess) e = launch_bwd_prep(g, dO, O, Ores, Q, K, V, Dv, emax, st);
  if (e == cudaSuccess) e = launch_bwd_main(g, plan, LSE, Dv, emax, mask, dQ, dK, dV, partial, status, st);
  if (e == cudaSuccess) e = launch_dbias_reduce_t(g, sp, partial, dBias, st);
  return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA;
}
