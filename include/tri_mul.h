/*
 * Triangle multiplicative update: gating and triangular contraction, forward
 * and backward, on one GB300 (sm_103a).
 *
 * What is computed (the fast_trimul article on kongchang.com, section
 * "什么是三角乘法更新": element-wise gating, an outer product of two gated
 * operands and a reduction along one axis of the N x N pair representation;
 * TurboPairFormer, arXiv 2610.05854v1, Abstract: the triangle multiplication
 * kernels run beside the triangle attention in training). For batch b, pair
 * position (i, j) and channel c, from four projections of the pair
 * representation, P_a, G_a, P_b, G_b:
 *
 *     a = sigmoid(G_a) * P_a,   b = sigmoid(G_b) * P_b      (rounded to BF16)
 *     outgoing: X[b,i,j,c] = sum_k a[b,i,k,c] * b[b,j,k,c]
 *     incoming: X[b,i,j,c] = sum_k a[b,k,i,c] * b[b,k,j,c]
 *
 * The gated operands are rounded to BF16 once; the contraction accumulates
 * in FP32 on the tensor cores. The surrounding layer norms, projections and
 * output gate are not part of this operation.
 *
 * Layouts (row-major, all tensors BF16 unless stated). X, dX and the saved
 * gated operands A, Bm are always channel-major, [B, C, N, N]. The
 * projections P_a, G_a, P_b, G_b and their gradients take shape.layout:
 *   TRI_MUL_LAYOUT_PAIR           [B, N, N, C], channels innermost (the pair
 *                                 representation's own layout). The gating
 *                                 kernel changes the layout: A[b,c,i,k] =
 *                                 a[b,i,k,c] (outgoing) or a[b,k,i,c]
 *                                 (incoming), likewise Bm, so that X[b,c] =
 *                                 A[b,c] Bm[b,c]^T in both directions; the
 *                                 backward pass goes through FP32 dA, dB in
 *                                 the workspace and a layout-changing
 *                                 gradient kernel.
 *   TRI_MUL_LAYOUT_CHANNEL_MAJOR  [B, C, N, N] (what a projection GEMM writes
 *                                 when it is asked for channel-major output).
 *                                 A[b,c,x,y] = a[b,x,y,c] in both directions;
 *                                 X[b,c] = A[b,c] Bm[b,c]^T (outgoing) or
 *                                 A[b,c]^T Bm[b,c] (incoming). The backward
 *                                 pass needs no workspace: the gating
 *                                 gradient runs in the contractions' epilogue.
 *
 * Accuracy: the gating runs in FP32 (fast exponential and reciprocal), accurate
 * to a few FP32 ulp plus about one ulp per unit of |G| before the BF16
 * rounding, for gate logits |G| < 87; below G = -87 the gated value is 0.
 *
 * Requirements: B >= 1, 16 <= N <= TRI_MUL_MAX_N with N a multiple of 8,
 * 8 <= C <= TRI_MUL_MAX_C with C a multiple of 8, B * C <= 65535, every
 * pointer 16-byte aligned and on the current device, tensors not
 * overlapping. Return codes are the TRI_ATTN_* codes of tri_attn.h; a call
 * that returns an error has enqueued nothing. Calls are asynchronous on
 * `stream` (a cudaStream_t, NULL = the legacy default stream) and
 * deterministic: every output element is computed in a fixed order,
 * independent of timing. Kernels never trap; a bounded device-side wait that
 * expires records TRI_ATTN_ERR_TIMEOUT for tri_attn_device_status(). With
 * tri_attn_set_timing_events(), the k-th event is recorded after the k-th
 * kernel of a call: forward 0 gating, 1 contraction; backward 0 the dA
 * contraction, 1 the dB contraction, and in the pair layout 2 the gating
 * gradient.
 */
#ifndef TRI_MUL_H
#define TRI_MUL_H

#include "tri_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define TRI_MUL_MAX_N 4096
#define TRI_MUL_MAX_C 1024

#define TRI_MUL_LAYOUT_PAIR 0          /* P, G and their gradients [B, N, N, C] */
#define TRI_MUL_LAYOUT_CHANNEL_MAJOR 1 /* P, G and their gradients [B, C, N, N] */

typedef struct tri_mul_shape {
    int B;        /* batch */
    int N;        /* residues: the pair representation is N x N */
    int C;        /* channels of the gated projections */
    int incoming; /* 0: outgoing edges (sum over the pair tensor's last position axis), 1: incoming (first axis) */
    int layout;   /* TRI_MUL_LAYOUT_PAIR or TRI_MUL_LAYOUT_CHANNEL_MAJOR */
} tri_mul_shape;

/*
 * Forward. Reads Pa, Ga, Pb, Gb (shape.layout). Writes the gated operands A
 * and Bm (channel-major; the backward pass reads them) and X (channel-major,
 * FP32 sums rounded to BF16). All buffers are owned by the caller.
 */
int tri_mul_fwd(tri_mul_shape shape, const tri_attn_bf16 *Pa, const tri_attn_bf16 *Ga,
                const tri_attn_bf16 *Pb, const tri_attn_bf16 *Gb, tri_attn_bf16 *A,
                tri_attn_bf16 *Bm, tri_attn_bf16 *X, void *stream);

/* Bytes of device workspace tri_mul_bwd needs: two FP32 [B, C, N, N] buffers in the pair layout,
 * none in the channel-major layout; 0 for a bad shape. */
size_t tri_mul_bwd_workspace_size(tri_mul_shape shape);

/*
 * Backward: gradients of sum(dX * X) with respect to Pa, Ga, Pb, Gb, taking
 * the BF16 rounding of the gated operands as the identity. Reads Pa, Ga, Pb,
 * Gb (shape.layout), A and Bm (as tri_mul_fwd wrote them) and dX
 * (channel-major). Writes dPa, dGa, dPb, dGb (shape.layout, BF16 of FP32
 * values): dP = dA sigmoid(G), dG = dA P sigmoid(G) (1 - sigmoid(G)), with
 * dA and dB the gradients of the gated operands, products of dX with Bm and
 * A summed in FP32. workspace: at least tri_mul_bwd_workspace_size(shape)
 * bytes of device memory, 16-byte aligned, else TRI_ATTN_ERR_WORKSPACE (may
 * be NULL when that size is 0).
 */
int tri_mul_bwd(tri_mul_shape shape, const tri_attn_bf16 *Pa, const tri_attn_bf16 *Ga,
                const tri_attn_bf16 *Pb, const tri_attn_bf16 *Gb, const tri_attn_bf16 *A,
                const tri_attn_bf16 *Bm, const tri_attn_bf16 *dX, tri_attn_bf16 *dPa,
                tri_attn_bf16 *dGa, tri_attn_bf16 *dPb, tri_attn_bf16 *dGb, void *workspace,
                size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TRI_MUL_H */
