/*
 * tri_attn.h - C ABI of the GB300 (sm_103a) triangle-attention library.
 *
 * Operation (TurboPairFormer: Fast and Stable Protein Folding Model Training
 * with an Optimized Triangle Attention Kernel, arXiv 2610.05854v1, Abstract):
 * every row-slice i of an N x N pair tensor runs multi-head attention over its
 * N positions, and a pair bias bias[b,h,j,k] is added to the scores of every
 * slice. Per batch b, slice i, head h, query j, key k:
 *
 *   S[j,k] = scale * <Q[b,i,j,h,:], K[b,i,k,h,:]> + bias[b,h,j,k] + mask[b,i,k]
 *   P      = softmax over k,   O[b,i,j,h,:] = sum_k P[j,k] V[b,i,k,h,:]
 *
 * The backward pass returns dQ, dK, dV and dBias = sum over slices of the
 * per-slice score gradient (the bias is shared by all slices, which adds that
 * reduction to the usual ones over queries and keys).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are dense, row-major, on the current CUDA device:
 *     Q K V O Ores dO dQ dK dV : BF16 pair tensors, [B, S, N, H, d] for the
 *                                starting node (slices along pair axis 1),
 *                                [B, N, S, H, d] for the ending node (slices
 *                                along pair axis 2); S = number of slices
 *     bias dBias               : BF16 [B, H, N, N]
 *     mask                     : BF16 [B, S, N], additive (0 or -inf), may be NULL
 *     LSE                      : FP32 [B, S, H, N], natural-log log-sum-exp of the
 *                                scores of each query row (-inf for a row whose
 *                                keys are all masked)
 * - Supported: d in {16, 32}; 1 <= N <= TRI_ATTN_MAX_N; 1 <= H <= TRI_ATTN_MAX_H;
 *   B, S >= 1. scale is
 *   any finite float (1/sqrt(d) is the usual choice).
 * - Input range: every input must be finite (mask entries 0 or -inf). The
 *   kernels stage Q, K, V and dO as FP16 tensor-core operands after multiplying
 *   each (batch, slice, head) block by a power of two chosen from the block's
 *   largest magnitude, and undo it exactly in FP32, so no BF16 magnitude is too
 *   large or too small as such: with the largest magnitude M of a block between
 *   2^-40 and 2^40, every entry of the block down to M * 2^-20 is staged exactly
 *   (smaller entries keep an absolute error below M * 2^-21, far under the BF16
 *   rounding of the results). Blocks whose M lies outside [2^-40, 2^40] lose
 *   precision gradually (the scale exponent is clamped to +-40); an all-zero
 *   block is exact. O, Ores and LSE given to the backward must be the forward's
 *   outputs for the same inputs.
 * - Every device pointer must be 16-byte aligned (TMA requirement).
 * - Ownership: the caller allocates and owns every buffer, including the
 *   backward workspace. The library allocates no device memory, never
 *   synchronises, and enqueues all work on `stream` (a cudaStream_t; NULL is
 *   the legacy default stream). Outputs are overwritten, never accumulated.
 * - Determinism: for a fixed shape on a fixed GPU model, every output is
 *   bitwise identical across calls. No floating-point atomics are used. The
 *   forward's reductions run in an order fixed by the shape; the backward
 *   splits its (head, slice) pairs over as many thread-block clusters as the
 *   device keeps resident at once, and its dBias summation order is fixed by
 *   the shape and that split (tri_attn_bwd_split reports it): a property of the
 *   GPU model and this library build, not of timing.
 * - Errors: each call returns TRI_ATTN_OK or a negative code. Arguments, the
 *   work split, tensor maps and the kernels' attributes are all checked on the
 *   host before the first kernel is enqueued, so a call that returns an error
 *   has launched nothing (TRI_ATTN_ERR_CUDA from the launches themselves
 *   excepted).
 * - First call per device: the first call of each entry point on a device does
 *   one-time host set-up there (kernel attributes, occupancy and device
 *   queries, symbol addresses); make it before capturing the stream into a
 *   CUDA graph.
 *   Kernels never trap: a bounded device-side wait that expires records
 *   TRI_ATTN_ERR_TIMEOUT in a device status word that
 *   tri_attn_device_status() reads.
 * - Ending-node attention (attention along the pair tensor's first axis, one
 *   slice per entry of its second axis) reads and writes the pair tensors in
 *   place with shape.node = TRI_ATTN_NODE_ENDING: no transposed copies.
 *   bias, mask, LSE and dBias keep the shapes above, in terms of the slices
 *   and positions of the attention that runs.
 */
#ifndef TRI_ATTN_H
#define TRI_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raw BF16 storage (IEEE binary32 with the low 16 bits dropped). */
typedef uint16_t tri_attn_bf16;

#define TRI_ATTN_MAX_N 1024
#define TRI_ATTN_MAX_H 256

/* Which pair axis holds the slices (shape.node). */
#define TRI_ATTN_NODE_STARTING 0 /* pair tensors [B, S, N, H, d] */
#define TRI_ATTN_NODE_ENDING 1   /* pair tensors [B, N, S, H, d] */

typedef struct tri_attn_shape {
    int B;       /* batch */
    int S;       /* slices of the pair tensor (N for a square pair tensor) */
    int N;       /* positions attended over inside a slice */
    int H;       /* heads */
    int d;       /* head dimension: 16 or 32 */
    float scale; /* multiplies Q.K only (not the bias) */
    int node;    /* TRI_ATTN_NODE_STARTING (0) or TRI_ATTN_NODE_ENDING (1) */
} tri_attn_shape;

enum {
    TRI_ATTN_OK = 0,
    TRI_ATTN_ERR_INVALID_ARG = -1,  /* NULL where required, non-positive or non-finite sizes, bad node */
    TRI_ATTN_ERR_UNSUPPORTED = -2,  /* d not 16/32, N above the limit, misaligned pointer */
    TRI_ATTN_ERR_WORKSPACE = -3,    /* workspace NULL or smaller than tri_attn_bwd_workspace_size */
    TRI_ATTN_ERR_CUDA = -4,         /* a CUDA runtime/driver call or launch failed */
    TRI_ATTN_ERR_TIMEOUT = -5,      /* a bounded device wait expired (see tri_attn_device_status) */
    TRI_ATTN_ERR_STATIC_TOO_SMALL = -6 /* tri_attn_bwd_static: shape needs more than the static workspace */
};

/* Human-readable text of a return code (static storage, never NULL). */
const char *tri_attn_strerror(int code);

/*
 * Forward pass (arXiv 2610.05854v1, Abstract: BF16 forward outputs plus the
 * output-residual that the backward correction uses).
 *
 * Inputs : Q, K, V, bias; mask may be NULL (no masking).
 * Outputs: O    = BF16 round-to-nearest of the FP32 attention output;
 *          LSE  = per-row log-sum-exp (FP32);
 *          Ores = BF16 round-to-nearest of (O_fp32 - O), the output-rounding
 *                 residual; may be NULL, in which case it is not written.
 * Writing Ores never changes O.
 */
int tri_attn_fwd(tri_attn_shape shape,
                 const tri_attn_bf16 *Q, const tri_attn_bf16 *K, const tri_attn_bf16 *V,
                 const tri_attn_bf16 *bias, const tri_attn_bf16 *mask,
                 tri_attn_bf16 *O, float *LSE, tri_attn_bf16 *Ores,
                 void *stream);

/*
 * Bytes of device workspace tri_attn_bwd needs for `shape` on the current
 * device (the bound on the work split depends on its SM count). Returns 0 for
 * an unsupported shape or when the device cannot be queried.
 */
size_t tri_attn_bwd_workspace_size(tri_attn_shape shape);

/*
 * The backward's work split on the current device: *clusters receives the
 * number of thread-block clusters its (head, slice) pairs are divided over
 * (cluster c takes the contiguous range [c W / n, (c + 1) W / n) of the
 * W = B*H*S pairs, head-major), *slots_per_head the most clusters that share
 * one head (the dBias partial slots per head). These two numbers and the shape
 * fix every summation order of the backward. static_entry != 0 reports the
 * split of tri_attn_bwd_static (which may use fewer clusters), else that of
 * tri_attn_bwd. Returns TRI_ATTN_OK, TRI_ATTN_ERR_INVALID_ARG /
 * TRI_ATTN_ERR_UNSUPPORTED for a bad shape or NULL outputs,
 * TRI_ATTN_ERR_STATIC_TOO_SMALL (static_entry only) or TRI_ATTN_ERR_CUDA.
 */
int tri_attn_bwd_split(tri_attn_shape shape, int static_entry, int *clusters, int *slots_per_head);

/*
 * Backward pass (arXiv 2610.05854v1, Abstract: key-tile-parallel backward that
 * recomputes each probability tile once, ordered partial reductions instead of
 * floating-point atomics, and the softmax correction D computed in FP32 from
 * the output plus its rounding residual).
 *
 * Inputs : Q, K, V, bias, mask (nullable) as given to tri_attn_fwd; O and LSE
 *          from tri_attn_fwd; Ores from tri_attn_fwd, or NULL for the
 *          uncompensated variant (D from the BF16 output alone); dO, the
 *          gradient of the loss with respect to O.
 * Outputs: dQ, dK, dV (BF16 [B,S,N,H,d]) and dBias (BF16 [B,H,N,N], summed over
 *          the S slices, not over the batch).
 * Workspace: `workspace` points to at least tri_attn_bwd_workspace_size(shape)
 *          bytes of device memory (16-byte aligned) that the call may overwrite;
 *          its contents on entry do not matter.
 */
int tri_attn_bwd(tri_attn_shape shape,
                 const tri_attn_bf16 *Q, const tri_attn_bf16 *K, const tri_attn_bf16 *V,
                 const tri_attn_bf16 *bias, const tri_attn_bf16 *mask,
                 const tri_attn_bf16 *O, const tri_attn_bf16 *Ores, const float *LSE,
                 const tri_attn_bf16 *dO,
                 tri_attn_bf16 *dQ, tri_attn_bf16 *dK, tri_attn_bf16 *dV, tri_attn_bf16 *dBias,
                 void *workspace, size_t workspace_bytes,
                 void *stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of the
 * current device: TRI_ATTN_OK, or TRI_ATTN_ERR_TIMEOUT if a bounded device wait
 * expired in any call since the last check (that call's outputs are invalid).
 * Returns TRI_ATTN_ERR_CUDA if the synchronisation itself fails.
 */
int tri_attn_device_status(void *stream);

/*
 * Backward pass that allocates nothing and takes no workspace argument.
 * (This entry point is a library convenience; the paper has no counterpart.)
 *
 * Some callers cannot allocate device memory when they call the backward pass:
 * a plugin whose host framework hands it only its input and output tensors and
 * owns every other byte of device memory, or a service that runs on a fixed,
 * pre-planned memory budget where a cudaMalloc at call time could fail or stall
 * the stream. For them, this call takes its scratch (the D correction, the
 * transposed bias and the dBias partials) from one array of
 * TRI_ATTN_STATIC_WORKSPACE_BYTES bytes that the library defines at file scope
 * in device memory; every GPU on which the library is loaded holds that array
 * until the process exits. The call itself allocates nothing.
 *
 * Arguments, layouts and outputs are exactly those of tri_attn_bwd minus the
 * workspace. The work is spread over fewer clusters when the dBias partial
 * slots of the full split do not fit in the array, so dBias may be summed in a
 * different (still fixed) order than tri_attn_bwd uses for the same shape, and
 * the call is slower; the results agree within rounding.
 * Returns TRI_ATTN_ERR_STATIC_TOO_SMALL, before enqueuing anything, when even
 * one slot per head does not fit (B = 1, H = 4, S = N = 768 fits with two slots
 * per head; S = N = 1024 does not).
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) besides the set-up every
 * backward call does once per device; make that first call before any stream
 * capture. Sharing: every call uses the same array and leaves its
 * contents behind. Nothing in it needs to start at zero (each call writes every
 * byte it reads first), but two calls whose kernels overlap on the GPU (other
 * streams, other host threads) race on the array and must be serialised by the
 * caller.
 */
#define TRI_ATTN_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)

int tri_attn_bwd_static(tri_attn_shape shape,
                        const tri_attn_bf16 *Q, const tri_attn_bf16 *K, const tri_attn_bf16 *V,
                        const tri_attn_bf16 *bias, const tri_attn_bf16 *mask,
                        const tri_attn_bf16 *O, const tri_attn_bf16 *Ores, const float *LSE,
                        const tri_attn_bf16 *dO,
                        tri_attn_bf16 *dQ, tri_attn_bf16 *dK, tri_attn_bf16 *dV, tri_attn_bf16 *dBias,
                        void *stream);

/*
 * Per-kernel timing instrumentation (off by default). After this call, every
 * tri_attn_fwd / tri_attn_bwd issued by the calling host thread records
 * events[k] (a cudaEvent_t created by the caller) on the call's stream right
 * after enqueuing the call's k-th kernel, for k < n. Kernel order:
 * tri_attn_fwd = {V scale pre-pass, forward}; tri_attn_bwd = {bias transpose,
 * preparation (D correction and operand scales), main backward, dBias
 * reduction}. events = NULL or n = 0 switches it off. The events stay
 * owned by the caller and must stay valid while instrumentation is on.
 * Returns TRI_ATTN_OK, or TRI_ATTN_ERR_INVALID_ARG for n < 0.
 */
int tri_attn_set_timing_events(void *const *events, int n);

#ifdef __cplusplus
}
#endif

#endif /* TRI_ATTN_H */
