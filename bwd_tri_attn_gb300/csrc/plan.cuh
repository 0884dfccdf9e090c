// Launch plans: everything a call needs that can fail on the host (tensor-map encoding, the
// kernels' one-time attribute set-up, the work split) is settled in a plan before the call
// enqueues its first kernel, so that a call that returns an error has launched nothing.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tri_attn.h"

namespace triattn {

struct FwdPlan {
  CUtensorMap mq, mk, mv, mb;
  int grid;  // persistent CTAs
};

struct BwdPlan {
  CUtensorMap mq, mk, mv, mdo, mbt, mdk, mdv;
  BwdSplit sp;
};

cudaError_t plan_fwd(const Dims &g, const uint16_t *Q, const uint16_t *K, const uint16_t *V, const uint16_t *bias,
                     FwdPlan *p);
cudaError_t launch_fwd_vscale(const Dims &g, const uint16_t *V, float *LSE, cudaStream_t stream);
cudaError_t launch_fwd(const Dims &g, const FwdPlan &p, const uint16_t *bias, const uint16_t *mask, uint16_t *O,
                       float *LSE, uint16_t *Ores, int *status, cudaStream_t stream);

// Tensor maps and attribute set-up of the main backward kernel (sp: the split already chosen).
cudaError_t plan_bwd(const Dims &g, const BwdSplit &sp, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     const uint16_t *dO, const uint16_t *biasT, uint16_t *dK, uint16_t *dV, BwdPlan *p);
// (also zeroes the per-(batch, head) exponent maxima emax[B*H][4] that launch_bwd_prep accumulates)
cudaError_t launch_bias_transpose(const Dims &g, const uint16_t *bias, uint16_t *biasT, int *emax,
                                  cudaStream_t stream);
cudaError_t launch_bwd_prep(const Dims &g, const uint16_t *dO, const uint16_t *O, const uint16_t *Ores,
                            const uint16_t *Q, const uint16_t *K, const uint16_t *V, float *Dout, int *emax,
                            cudaStream_t stream);
cudaError_t launch_bwd_main(const Dims &g, const BwdPlan &p, const float *LSE, const float *Dv, const int *emax,
                            const uint16_t *mask, uint16_t *dQ, uint16_t *dK, uint16_t *dV, float *partial,
                            int *status, cudaStream_t stream);
cudaError_t launch_dbias_reduce_t(const Dims &g, const BwdSplit &sp, const float *partial, uint16_t *dBias,
                                  cudaStream_t stream);

// A checked and planned attention call, ready to enqueue (entry points of other files, such as
// the surrounding block, prepare every call before they launch anything).
struct AttnFwdCall {
  Dims g;
  FwdPlan plan;
  const uint16_t *V, *bias, *mask;
  uint16_t *O, *Ores;
  float *LSE;
  int *status;
};

struct AttnBwdCall {
  Dims g;
  BwdSplit sp;
  BwdPlan plan;
  const uint16_t *Q, *K, *V, *bias, *mask, *O, *Ores, *dO;
  const float *LSE;
  uint16_t *dQ, *dK, *dV, *dBias, *biasT;
  float *Dv, *partial;
  int *emax, *status;
};

int attn_fwd_prepare(const tri_attn_shape &shape, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     const uint16_t *bias, const uint16_t *mask, uint16_t *O, float *LSE, uint16_t *Ores,
                     AttnFwdCall *c);
cudaError_t attn_fwd_enqueue(const AttnFwdCall &c, int mark0, cudaStream_t st);
int attn_bwd_prepare(const tri_attn_shape &shape, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     const uint16_t *bias, const uint16_t *mask, const uint16_t *O, const uint16_t *Ores,
                     const float *LSE, const uint16_t *dO, uint16_t *dQ, uint16_t *dK, uint16_t *dV,
                     uint16_t *dBias, void *workspace, size_t workspace_bytes, AttnBwdCall *c);
cudaError_t attn_bwd_enqueue(const AttnBwdCall &c, int mark0, cudaStream_t st);
cudaError_t timing_mark(int k, cudaStream_t st);

cudaError_t device_sm_count(int *nsm);
cudaError_t bwd_split_active(const Dims &g, BwdSplit *sp);
int bwd_slots_for(const Dims &g, int NC);
int bwd_slots_max(const Dims &g, int nsm);
int *device_status_word();

}  // namespace triattn
