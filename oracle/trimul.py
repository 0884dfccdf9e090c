"""FP64 CPU oracle for the triangle multiplicative update (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this module. The CUDA library never loads it, and the
two share no code.

What it computes (the fast_trimul article, section "什么是三角乘法更新": the
update combines element-wise gating, a matrix outer product and a reduction
along one axis of the N x N pair representation; TurboPairFormer, arXiv
2610.05854v1, Abstract, last sentence: the triangle multiplication kernels that
run next to the attention in training). Written out, per batch b, pair
position (i, j) and channel c, with the projections P_a, G_a, P_b, G_b of the
pair representation given ([B, N, N, C]):

    a = sigmoid(G_a) * P_a,   b = sigmoid(G_b) * P_b         (element-wise gating)
    outgoing:  X[b,i,j,c] = sum_k a[b,i,k,c] * b[b,j,k,c]    (row i of a against row j of b)
    incoming:  X[b,i,j,c] = sum_k a[b,k,i,c] * b[b,k,j,c]    (column i against column j)

The gated operands are stored in BF16 (round to nearest even) before the
contraction, as in a BF16 training pipeline; the contraction itself is exact
here (FP64). The backward pass returns the gradients of L = sum(dX * X) with
respect to P_a, G_a, P_b, G_b, taking the BF16 storage of a and b as the
identity (as autograd does for a dtype cast).
"""
from __future__ import annotations

import numpy as np


def _f64(t) -> np.ndarray:
    if hasattr(t, "detach"):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest BF16 value (ties to even), returned as float64."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16).double().numpy()


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def gated(p, g, bf16: bool = True) -> np.ndarray:
    """sigmoid(g) * p, stored in BF16 unless bf16 is False."""
    a = sigmoid(_f64(g)) * _f64(p)
    return round_bf16(a) if bf16 else a


def contract(a: np.ndarray, b: np.ndarray, incoming: bool) -> np.ndarray:
    """X of the outgoing / incoming update from the gated operands ([B, N, N, C] each)."""
    if incoming:
        return np.einsum("bkic,bkjc->bijc", a, b)
    return np.einsum("bikc,bjkc->bijc", a, b)


def fwd(pa, ga, pb, gb, incoming: bool = False, bf16: bool = True):
    """Returns X [B, N, N, C] (float64)."""
    return contract(gated(pa, ga, bf16), gated(pb, gb, bf16), incoming)


def bwd(pa, ga, pb, gb, dX, incoming: bool = False, bf16: bool = True):
    """Gradients of sum(dX * X) with respect to P_a, G_a, P_b, G_b ([B, N, N, C] float64 each)."""
    pa, ga, pb, gb, dX = (_f64(t) for t in (pa, ga, pb, gb, dX))
    a, b = gated(pa, ga, bf16), gated(pb, gb, bf16)
    if incoming:
        da = np.einsum("bijc,bkjc->bkic", dX, b)  # dX[i,j] b[k,j] -> dA[k,i]
        db = np.einsum("bijc,bkic->bkjc", dX, a)  # dX[i,j] a[k,i] -> dB[k,j]
    else:
        da = np.einsum("bijc,bjkc->bikc", dX, b)  # dX[i,j] b[j,k] -> dA[i,k]
        db = np.einsum("bijc,bikc->bjkc", dX, a)  # dX[i,j] a[i,k] -> dB[j,k]
    sa, sb = sigmoid(ga), sigmoid(gb)
    return {"dPa": da * sa, "dGa": da * pa * sa * (1.0 - sa), "dPb": db * sb, "dGb": db * pb * sb * (1.0 - sb)}
