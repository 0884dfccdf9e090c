// Host side of the C ABI declared in include/tri_attn.h: argument checks,
// workspace layout and kernel launches. No device memory is allocated here and
// nothing synchronises except tri_attn_device_status().
#include <math.h>
#include <mutex>

#include "common.cuh"

#include "plan.cuh"

namespace triattn {
int static_bwd_split(const tri_attn_shape &s, BwdSplit *sp);
}  // namespace triattn

using namespace triattn;

// Device status word: bounded waits that expire store a nonzero code here.
__device__ int g_tri_attn_status;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const tri_attn_shape &s) {
  if (s.B < 1 || s.S < 1 || s.N < 1 || s.H < 1 || !isfinite(s.scale)) return TRI_ATTN_ERR_INVALID_ARG;
  if (s.node != TRI_ATTN_NODE_STARTING && s.node != TRI_ATTN_NODE_ENDING) return TRI_ATTN_ERR_INVALID_ARG;
  if (s.d != 16 && s.d != 32) return TRI_ATTN_ERR_UNSUPPORTED;
  if (s.N > TRI_ATTN_MAX_N || s.H > TRI_ATTN_MAX_H) return TRI_ATTN_ERR_UNSUPPORTED;
  // grid dimensions and 32-bit tile coordinates
  if ((int64_t)s.B * s.S > 65535 || (int64_t)s.B * s.H * s.S > (1ll << 30)) return TRI_ATTN_ERR_UNSUPPORTED;
  return TRI_ATTN_OK;
}

Dims to_dims(const tri_attn_shape &s) { return Dims{s.B, s.S, s.N, s.H, s.d, s.scale, s.node}; }

// Backward workspace: the FP32 correction D [B,S,H,N], the operand exponent maxima
// int [B,H][4], the transposed and tile-padded BF16 bias [B*H][NP][NP] (NP = N
// rounded up to 128), and the FP32 dBias partials [B*H][slots][NP][NP]: one slot
// per cluster that works on a head.
struct WorkspaceLayout {
  size_t d_off, scl_off, biast_off, partial_off, total;
  int slots;
};

// Workspace layout for the current device (nsm: its SM count, which bounds the split).
WorkspaceLayout layout_for(const tri_attn_shape &s, int nsm) {
  WorkspaceLayout w;
  const Dims g = to_dims(s);
  const size_t NP = (size_t)(s.N + 127) / 128 * 128;
  const size_t rows = (size_t)s.B * s.S * s.H * s.N;
  w.slots = bwd_slots_max(g, nsm);
  w.d_off = 0;
  w.scl_off = align_up(sizeof(float) * rows);
  w.biast_off = w.scl_off + align_up(16 * (size_t)s.B * s.H);
  w.partial_off = w.biast_off + align_up(2 * (size_t)s.B * s.H * NP * NP);
  w.total = w.partial_off + align_up(sizeof(float) * (size_t)w.slots * s.B * s.H * NP * NP);
  return w;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? TRI_ATTN_OK : TRI_ATTN_ERR_CUDA; }

// Device address of the status word on the current device (looked up once per device).
int *status_word() {
  static std::mutex mu;
  static int *addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tri_attn_status) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int *>(p);
  }
  return addr[dev];
}

// Optional per-kernel timing events of the calling host thread.
thread_local void *const *t_events = nullptr;
thread_local int t_nevents = 0;

// Records the caller's k-th timing event after the k-th kernel of a call.
cudaError_t mark(int k, cudaStream_t st) {
  if (t_events && k < t_nevents) return cudaEventRecord(static_cast<cudaEvent_t>(t_events[k]), st);
  return cudaSuccess;
}

}  // namespace

namespace triattn {
// Status word of the current device, for entry points defined in other files.
int *device_status_word() { return status_word(); }
// The calling thread's k-th timing event, for entry points defined in other files.
cudaError_t timing_mark(int k, cudaStream_t st) { return mark(k, st); }

// Every check and the launch plan of a forward call, with nothing enqueued.
int attn_fwd_prepare(const tri_attn_shape &shape, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     const uint16_t *bias, const uint16_t *mask, uint16_t *O, float *LSE, uint16_t *Ores,
                     AttnFwdCall *c) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!Q || !K || !V || !bias || !O || !LSE) return TRI_ATTN_ERR_INVALID_ARG;
  const void *ptrs[] = {Q, K, V, bias, mask, O, LSE, Ores};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return TRI_ATTN_ERR_UNSUPPORTED;
  c->g = to_dims(shape);
  c->V = V;
  c->bias = bias;
  c->mask = mask;
  c->O = O;
  c->LSE = LSE;
  c->Ores = Ores;
  c->status = status_word();
  if (!c->status) return TRI_ATTN_ERR_CUDA;
  if (plan_fwd(c->g, Q, K, V, bias, &c->plan) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  return TRI_ATTN_OK;
}

// The forward's kernels; the caller's timing events mark0, mark0 + 1 follow them.
cudaError_t attn_fwd_enqueue(const AttnFwdCall &c, int mark0, cudaStream_t st) {
  cudaError_t e = launch_fwd_vscale(c.g, c.V, c.LSE, st);
  if (e == cudaSuccess) e = mark(mark0, st);
  if (e == cudaSuccess) e = launch_fwd(c.g, c.plan, c.bias, c.mask, c.O, c.LSE, c.Ores, c.status, st);
  if (e == cudaSuccess) e = mark(mark0 + 1, st);
  return e;
}

// Every check, the work split and the launch plan of a backward call, with nothing enqueued.
int attn_bwd_prepare(const tri_attn_shape &shape, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     const uint16_t *bias, const uint16_t *mask, const uint16_t *O, const uint16_t *Ores,
                     const float *LSE, const uint16_t *dO, uint16_t *dQ, uint16_t *dK, uint16_t *dV,
                     uint16_t *dBias, void *workspace, size_t workspace_bytes, AttnBwdCall *c) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!Q || !K || !V || !bias || !O || !LSE || !dO || !dQ || !dK || !dV || !dBias)
    return TRI_ATTN_ERR_INVALID_ARG;
  const void *ptrs[] = {Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias, workspace};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return TRI_ATTN_ERR_UNSUPPORTED;
  int nsm = 0;
  if (device_sm_count(&nsm) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  const WorkspaceLayout w = layout_for(shape, nsm);
  if (!workspace || workspace_bytes < w.total) return TRI_ATTN_ERR_WORKSPACE;
  c->g = to_dims(shape);
  // the work split (and with it the reduction order) is settled before anything is enqueued
  if (bwd_split_active(c->g, &c->sp) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  if (c->sp.KMAX > w.slots) return TRI_ATTN_ERR_CUDA;  // (cannot happen: the workspace covers every split)
  char *ws = static_cast<char *>(workspace);
  c->Dv = reinterpret_cast<float *>(ws + w.d_off);
  c->emax = reinterpret_cast<int *>(ws + w.scl_off);
  c->biasT = reinterpret_cast<uint16_t *>(ws + w.biast_off);
  c->partial = reinterpret_cast<float *>(ws + w.partial_off);
  c->Q = Q;
  c->K = K;
  c->V = V;
  c->bias = bias;
  c->mask = mask;
  c->O = O;
  c->Ores = Ores;
  c->LSE = LSE;
  c->dO = dO;
  c->dQ = dQ;
  c->dK = dK;
  c->dV = dV;
  c->dBias = dBias;
  c->status = status_word();
  if (!c->status) return TRI_ATTN_ERR_CUDA;
  if (plan_bwd(c->g, c->sp, Q, K, V, dO, c->biasT, dK, dV, &c->plan) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  return TRI_ATTN_OK;
}

// The backward's four kernels; the caller's timing events mark0 .. mark0 + 3 follow them.
cudaError_t attn_bwd_enqueue(const AttnBwdCall &c, int mark0, cudaStream_t st) {
  cudaError_t e = launch_bias_transpose(c.g, c.bias, c.biasT, c.emax, st);
  if (e == cudaSuccess) e = mark(mark0, st);
  if (e == cudaSuccess) e = launch_bwd_prep(c.g, c.dO, c.O, c.Ores, c.Q, c.K, c.V, c.Dv, c.emax, st);
  if (e == cudaSuccess) e = mark(mark0 + 1, st);
  if (e == cudaSuccess)
    e = launch_bwd_main(c.g, c.plan, c.LSE, c.Dv, c.emax, c.mask, c.dQ, c.dK, c.dV, c.partial, c.status, st);
  if (e == cudaSuccess) e = mark(mark0 + 2, st);
  if (e == cudaSuccess) e = launch_dbias_reduce_t(c.g, c.sp, c.partial, c.dBias, st);
  if (e == cudaSuccess) e = mark(mark0 + 3, st);
  return e;
}
}  // namespace triattn

extern "C" {

const char *tri_attn_strerror(int code) {
  switch (code) {
    case TRI_ATTN_OK: return "success";
    case TRI_ATTN_ERR_INVALID_ARG: return "invalid argument (NULL pointer, non-positive size, non-finite scale or unknown node)";
    case TRI_ATTN_ERR_UNSUPPORTED: return "unsupported configuration (d must be 16 or 32, N <= TRI_ATTN_MAX_N, H <= TRI_ATTN_MAX_H, pointers 16-byte aligned)";
    case TRI_ATTN_ERR_WORKSPACE: return "workspace missing or smaller than tri_attn_bwd_workspace_size()";
    case TRI_ATTN_ERR_CUDA: return "CUDA runtime error";
    case TRI_ATTN_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case TRI_ATTN_ERR_STATIC_TOO_SMALL:
      return "the shape needs more scratch than the library's static workspace (TRI_ATTN_STATIC_WORKSPACE_BYTES) holds";
    default: return "unknown error code";
  }
}

int tri_attn_fwd(tri_attn_shape shape, const tri_attn_bf16 *Q, const tri_attn_bf16 *K,
                 const tri_attn_bf16 *V, const tri_attn_bf16 *bias, const tri_attn_bf16 *mask,
                 tri_attn_bf16 *O, float *LSE, tri_attn_bf16 *Ores, void *stream) {
  AttnFwdCall c;
  const int rc = attn_fwd_prepare(shape, Q, K, V, bias, mask, O, LSE, Ores, &c);
  if (rc) return rc;
  return cuda_rc(attn_fwd_enqueue(c, 0, static_cast<cudaStream_t>(stream)));
}

size_t tri_attn_bwd_workspace_size(tri_attn_shape shape) {
  int nsm = 0;
  if (check_shape(shape) || device_sm_count(&nsm) != cudaSuccess) return 0;
  return layout_for(shape, nsm).total;
}

int tri_attn_bwd_split(tri_attn_shape shape, int static_entry, int *clusters, int *slots_per_head) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (!clusters || !slots_per_head) return TRI_ATTN_ERR_INVALID_ARG;
  BwdSplit sp;
  if (static_entry) {
    rc = static_bwd_split(shape, &sp);
    if (rc) return rc;
  } else if (bwd_split_active(to_dims(shape), &sp) != cudaSuccess) {
    return TRI_ATTN_ERR_CUDA;
  }
  *clusters = sp.NC;
  *slots_per_head = sp.KMAX;
  return TRI_ATTN_OK;
}

int tri_attn_bwd(tri_attn_shape shape, const tri_attn_bf16 *Q, const tri_attn_bf16 *K,
                 const tri_attn_bf16 *V, const tri_attn_bf16 *bias, const tri_attn_bf16 *mask,
                 const tri_attn_bf16 *O, const tri_attn_bf16 *Ores, const float *LSE,
                 const tri_attn_bf16 *dO, tri_attn_bf16 *dQ, tri_attn_bf16 *dK, tri_attn_bf16 *dV,
                 tri_attn_bf16 *dBias, void *workspace, size_t workspace_bytes, void *stream) {
  AttnBwdCall c;
  const int rc = attn_bwd_prepare(shape, Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias, workspace,
                                  workspace_bytes, &c);
  if (rc) return rc;
  return cuda_rc(attn_bwd_enqueue(c, 0, static_cast<cudaStream_t>(stream)));
}

int tri_attn_set_timing_events(void *const *events, int n) {
  if (n < 0) return TRI_ATTN_ERR_INVALID_ARG;
  t_events = (n > 0) ? events : nullptr;
  t_nevents = (events != nullptr) ? n : 0;
  return TRI_ATTN_OK;
}

int tri_attn_device_status(void *stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tri_attn_status, sizeof(int)) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_tri_attn_status, &zero, sizeof(int)) != cudaSuccess) return TRI_ATTN_ERR_CUDA;
    return TRI_ATTN_ERR_TIMEOUT;
  }
  return TRI_ATTN_OK;
}

}  // extern "C"
