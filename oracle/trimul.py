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


def sampled(pa, ga, pb, gb, dX, idx, incoming: bool = False, bf16: bool = True):
    """X and the four gradients at chosen entries only, for sizes where the full tensors are too
    large: idx is a list of (b, x, y, c). X is evaluated at [b, x, y, c] (its own index), each
    gradient at the projection entry [b, x, y, c]; dX is given in the pair layout [B, N, N, C].
    Every value is the definition written out for that one entry (an N-term dot product of gated
    rows or columns), so only the rows and columns it touches are gated.
    Returns a dict of float64 arrays with one value per entry."""
    pa, ga, pb, gb, dX = (_f64(t) for t in (pa, ga, pb, gb, dX))
    out = {k: [] for k in ("X", "dPa", "dGa", "dPb", "dGb")}
    for b, x, y, c in idx:
        # X[b,x,y,c]: outgoing sum_k a[x,k] b[y,k]; incoming sum_k a[k,x] b[k,y]
        if incoming:
            ar, br = gated(pa[b, :, x, c], ga[b, :, x, c], bf16), gated(pb[b, :, y, c], gb[b, :, y, c], bf16)
        else:
            ar, br = gated(pa[b, x, :, c], ga[b, x, :, c], bf16), gated(pb[b, y, :, c], gb[b, y, :, c], bf16)
        out["X"].append(float(np.dot(ar, br)))
        # gradient of the gated operand a at entry [x, y] (pair indices of the projection):
        # outgoing: a[x, y] meets b[j, y] in X[x, j] -> dA = sum_j dX[x, j] b[j, y]
        # incoming: a[x, y] meets b[x, j] in X[y, j] -> dA = sum_j dX[y, j] b[x, j]
        if incoming:
            da = float(np.dot(dX[b, y, :, c], gated(pb[b, x, :, c], gb[b, x, :, c], bf16)))
            # b[x, y] meets a[x, i] in X[i, y] -> dB = sum_i dX[i, y] a[x, i]
            db = float(np.dot(dX[b, :, y, c], gated(pa[b, x, :, c], ga[b, x, :, c], bf16)))
        else:
            da = float(np.dot(dX[b, x, :, c], gated(pb[b, :, y, c], gb[b, :, y, c], bf16)))
            # b[x, y] meets a[i, y] in X[i, x] -> dB = sum_i dX[i, x] a[i, y]
            db = float(np.dot(dX[b, :, x, c], gated(pa[b, :, y, c], ga[b, :, y, c], bf16)))
        sa, sb = sigmoid(ga[b, x, y, c]), sigmoid(gb[b, x, y, c])
        out["dPa"].append(da * sa)
        out["dGa"].append(da * pa[b, x, y, c] * sa * (1.0 - sa))
        out["dPb"].append(db * sb)
        out["dGb"].append(db * pb[b, x, y, c] * sb * (1.0 - sb))
    return {k: np.asarray(v) for k, v in out.items()}
