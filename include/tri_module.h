/*
 * Triangle-attention block around the attention core: LayerNorm, the q/k/v,
 * pair-bias and gate projections, the attention (tri_attn.h), the sigmoid gate
 * and the output projection, forward and backward, on one GB300 (sm_103a).
 *
 * What is computed. TurboPairFormer (arXiv 2610.05854v1, Abstract, first
 * sentence) places triangular attention in "AlphaFold3-style" models and
 * describes no layer around it; this block is the plainest reading of that
 * model family's triangle-attention layer. For a pair representation z
 * [B, N, N, c] and every pair position (x, y):
 *
 *     zt   = (z - mean) / sqrt(var + eps) * gamma + beta    (over the c channels, biased variance)
 *     q | k | v | gl = zt W^T                              (W: [4 H d, c], rows q, k, v, gate; no biases)
 *     bias[b, h, x, y] = zt[b, x, y, :] . wb[h, :]          (wb: [H, c])
 *     O    = tri_attn(q, k, v, bias, mask), scale 1/sqrt(d)
 *     out  = (sigmoid(gl) * O) Wo^T                         (Wo: [c, H d]; heads flattened h d + e)
 *
 * Starting node: slices along the first pair axis (q, k, v, O are the
 * attention's [B, S, N, H, d] tensors as they stand). Ending node: the same
 * block on the pair representation with its two pair axes swapped, the output
 * swapped back; no transposed copy is made: the attention reads the
 * projections in its ending-node layout, and the pair bias is written
 * transposed (bias[b, h, x, y] = zt[b, y, x, :] . wb[h, :]). The mask keeps
 * the attention's convention: additive BF16 [B, slice, key], or NULL.
 *
 * Precision: z, out, dout, dz, W, wb, Wo and every stored intermediate are BF16
 * (round to nearest even); LayerNorm statistics, gamma, beta and all five
 * weight gradients are FP32; every sum is accumulated in FP32, GEMMs on the
 * tensor cores with BF16 operands.
 *
 * Requirements: B >= 1, 16 <= N <= TRI_ATTN_MAX_N, c in {64, 128, 256},
 * d in {16, 32}, 1 <= H <= 8 with H * d a multiple of 64, B * N <= 65535, eps > 0
 * finite, every pointer 16-byte aligned and on the current device, buffers not
 * overlapping. Return codes are the TRI_ATTN_* codes of tri_attn.h; a call that
 * returns an error has enqueued nothing. Calls are asynchronous on `stream`
 * (a cudaStream_t, NULL = the legacy default stream) and deterministic for a
 * fixed shape and GPU model: every reduction (the attention's, the weight
 * gradients' sums over positions, the LayerNorm parameter gradients) runs in a
 * fixed order. Kernels never trap; a bounded device wait that expires records
 * TRI_ATTN_ERR_TIMEOUT for tri_attn_device_status(). The first call of each
 * entry point on a device does one-time host set-up (kernel attributes, the
 * attention backward's occupancy query); make it before any stream capture.
 *
 * Timing: with tri_attn_set_timing_events(), the k-th event is recorded after
 * the k-th kernel of a call. Forward: 0 LayerNorm and pair bias, 1 input
 * projections, 2 the attention's V-scale pre-pass, 3 the attention, 4 gate,
 * 5 output projection. Backward: 0 output-projection gradient with the gate
 * gradient, 1 Wo gradient partial sums, 2 their reduction, 3-6 the attention
 * backward (bias transpose, preparation, main kernel, dBias reduction),
 * 7 projection gradient dzt, 8 LayerNorm backward, 9 reduction of the
 * LayerNorm and bias-weight partial sums, 10 W gradient partial sums, 11 their
 * reduction.
 */
#ifndef TRI_MODULE_H
#define TRI_MODULE_H

#include "tri_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tri_module_shape {
    int B;     /* batch */
    int N;     /* residues: the pair representation is N x N */
    int c;     /* pair channels: 64, 128 or 256 */
    int H;     /* heads */
    int d;     /* head dimension: 16 or 32 */
    int node;  /* TRI_ATTN_NODE_STARTING (0) or TRI_ATTN_NODE_ENDING (1) */
    float eps; /* LayerNorm epsilon */
} tri_module_shape;

/*
 * Bytes of the activations the forward pass keeps for the backward pass (one
 * device buffer, layout private to the library: zt, the LayerNorm statistics,
 * q, k, v, gl, the pair bias, O, its rounding residual, the log-sum-exp and
 * the gated output); 0 for a bad shape.
 */
size_t tri_module_saved_size(tri_module_shape shape);

/*
 * Bytes of device workspace tri_module_bwd needs for `shape` on the current
 * device (it includes the attention backward's workspace, whose size depends on
 * the device's SM count). Returns 0 for an unsupported shape or when the device
 * cannot be queried.
 */
size_t tri_module_bwd_workspace_size(tri_module_shape shape);

/*
 * Forward. Reads z [B, N, N, c], gamma, beta [c] (FP32), W [4 H d, c],
 * wb [H, c], Wo [c, H d] and mask (NULL or [B, N, N]); writes out
 * [B, N, N, c] and fills `saved` (at least tri_module_saved_size() bytes, else
 * TRI_ATTN_ERR_WORKSPACE). All buffers are owned by the caller.
 */
int tri_module_fwd(tri_module_shape shape, const tri_attn_bf16 *z, const float *gamma, const float *beta,
                   const tri_attn_bf16 *W, const tri_attn_bf16 *wb, const tri_attn_bf16 *Wo,
                   const tri_attn_bf16 *mask, tri_attn_bf16 *out, void *saved, size_t saved_bytes,
                   void *stream);

/*
 * Backward: gradients of sum(dout * out). Reads the forward's inputs, `saved`
 * as tri_module_fwd left it, and dout [B, N, N, c]; writes dz [B, N, N, c]
 * (BF16), dgamma, dbeta [c], dW [4 H d, c], dwb [H, c], dWo [c, H d] (FP32,
 * overwritten, not accumulated). workspace: at least
 * tri_module_bwd_workspace_size() bytes, else TRI_ATTN_ERR_WORKSPACE.
 */
int tri_module_bwd(tri_module_shape shape, const tri_attn_bf16 *z, const float *gamma, const float *beta,
                   const tri_attn_bf16 *W, const tri_attn_bf16 *wb, const tri_attn_bf16 *Wo,
                   const tri_attn_bf16 *mask, const void *saved, size_t saved_bytes,
                   const tri_attn_bf16 *dout, tri_attn_bf16 *dz, float *dgamma, float *dbeta, float *dW,
                   float *dwb, float *dWo, void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TRI_MODULE_H */
