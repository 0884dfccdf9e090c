"""FP64 CPU oracle for the triangle-attention module around the attention core (test
infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline leg may
import this module. The CUDA library never loads it, and the two share no code.

What it computes. TurboPairFormer (arXiv 2610.05854v1, Abstract, first sentence) places
triangular attention inside "AlphaFold3-style" models and says nothing more about the layers
around it. The plainest reading is the triangle-attention block of that model family, the one
the pages' attention core sits in: per pair position of the pair representation z [B, N, N, c]

    zt    = LayerNorm(z) * gamma + beta                  (over the c channels, biased variance, eps)
    q|k|v|gl = zt W^T                                    (W [4 H d, c]: rows q, then k, v, gate; no biases)
    bias[b, h, x, y] = zt[b, x, y, :] . wb[h]            (wb [H, c]; the pair bias shared by all slices)
    O     = attention(q, k, v, bias, mask)               (starting node: slice = first pair axis)
    go    = sigmoid(gl) * O                              (heads flattened, channel h d + e)
    out   = go Wo^T                                      (Wo [c, H d])

The ending node is the same block applied to the pair representation with its two pair axes
swapped (z -> z^T), the result swapped back; the mask keeps the attention's own convention
([B, slice, key] in that frame). The attention step is the oracle's attention
(oracle.fwd / oracle.bwd), itself pinned against the pages' definition.

With bf16=True the oracle rounds to BF16 (nearest even) every tensor that a BF16 training
pipeline stores between the steps: zt, q, k, v, gl, bias, O, go and out in the forward pass;
dO (the attention's output gradient), the gate-logit gradient, the attention's four gradients
and dz in the backward pass. Derivatives take those roundings as the identity (as autograd
does for a dtype cast). With bf16=False every step is exact in FP64: the definition.
"""
from __future__ import annotations

import numpy as np

import oracle as attn


def _f64(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest BF16 value (ties to even), directly from float64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    # BF16 keeps the top 8 significand bits of a binary32 value. Rounding a double straight to
    # that precision: scale by the power of two of each value's binade so that the BF16 ulp is 1,
    # round half to even with numpy, scale back. Values below the BF16 normal range round on the
    # fixed subnormal grid (ulp 2^-133); overflow goes to +-inf.
    ax = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
        # log2 can be off by one next to a power of two: correct it exactly
        e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
        e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
        e = np.maximum(e, -126)
        ulp_exp = (e - 7).astype(np.int64)
        r = np.ldexp(np.round(np.ldexp(x, -ulp_exp)), ulp_exp)
        r = np.where(np.abs(r) > 3.3895313892515355e38, np.sign(x) * np.inf, r)
    return np.where(ax > 0, r, x)


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def layer_norm(z: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float):
    """(zt, mean, rstd): LayerNorm over the last axis with the biased variance."""
    mu = z.mean(axis=-1, keepdims=True)
    var = ((z - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    return (z - mu) * rstd * gamma + beta, mu[..., 0], rstd[..., 0]


def _frame(x, node):
    """The pair tensor in the frame where slices run along the first pair axis."""
    return x if node == 0 else np.ascontiguousarray(np.swapaxes(x, 1, 2))


def fwd(z, gamma, beta, W, wb, Wo, mask, H: int, d: int, node: int = 0, eps: float = 1e-5, bf16: bool = False):
    """Forward pass of the block. Returns a dict with out [B, N, N, c] and the intermediates
    (in the slice frame: zt, q, k, v [B, N, N, H, d], gl, bias [B, H, N, N], O, LSE, go)."""
    rb = round_bf16 if bf16 else (lambda a: a)
    z, gamma, beta, W, wb, Wo, mask = (_f64(t) for t in (z, gamma, beta, W, wb, Wo, mask))
    zf = _frame(z, node)
    B, N, _, c = zf.shape
    hd = H * d
    zt, mu, rstd = layer_norm(zf, gamma, beta, eps)
    zt = rb(zt)
    proj = zt @ W.T
    q, k, v, gl = (rb(proj[..., s * hd:(s + 1) * hd]) for s in range(4))
    bias = rb(np.einsum("bxyc,hc->bhxy", zt, wb))
    shp = (B, N, N, H, d)
    O, LSE = attn.fwd(q.reshape(shp), k.reshape(shp), v.reshape(shp), bias, mask)
    O = rb(O.reshape(B, N, N, hd))
    go = rb(sigmoid(gl) * O)
    out = rb(go @ Wo.T)
    return {"out": _frame(out, node), "zt": zt, "mu": mu, "rstd": rstd, "q": q, "k": k, "v": v, "gl": gl,
            "bias": bias, "O": O, "LSE": LSE, "go": go}


def bwd(z, gamma, beta, W, wb, Wo, mask, dout, H: int, d: int, node: int = 0, eps: float = 1e-5,
        bf16: bool = False):
    """Gradients of L = sum(dout * out) with respect to z, gamma, beta, W, wb and Wo."""
    rb = round_bf16 if bf16 else (lambda a: a)
    f = fwd(z, gamma, beta, W, wb, Wo, mask, H, d, node, eps, bf16)
    z, gamma, beta, W, wb, Wo, mask, dout = (_f64(t) for t in (z, gamma, beta, W, wb, Wo, mask, dout))
    zf, dof = _frame(z, node), _frame(dout, node)
    B, N, _, c = zf.shape
    hd = H * d
    # output projection and gate
    dWo = np.einsum("bxyc,bxyj->cj", dof, f["go"])
    dgo = dof @ Wo
    s = sigmoid(f["gl"])
    dO = rb(dgo * s)
    dgl = rb(dgo * f["O"] * s * (1.0 - s))
    # attention (the oracle's own backward: exact O, D = rowsum(dO * O))
    shp = (B, N, N, H, d)
    g = attn.bwd(f["q"].reshape(shp), f["k"].reshape(shp), f["v"].reshape(shp), f["bias"], mask, dO.reshape(shp))
    dq, dk, dv = (rb(g[n].reshape(B, N, N, hd)) for n in ("dQ", "dK", "dV"))
    dbias = rb(g["dBias"])
    # projections
    dproj = np.concatenate([dq, dk, dv, dgl], axis=-1)
    dW = np.einsum("bxyr,bxyc->rc", dproj, f["zt"])
    dwb = np.einsum("bhxy,bxyc->hc", dbias, f["zt"])
    dzt = dproj @ W + np.einsum("bhxy,hc->bxyc", dbias, wb)
    # layer norm
    zhat = (zf - f["mu"][..., None]) * f["rstd"][..., None]
    dgamma = np.einsum("bxyc,bxyc->c", dzt, zhat)
    dbeta = dzt.sum(axis=(0, 1, 2))
    dzh = dzt * gamma
    dz = f["rstd"][..., None] * (dzh - dzh.mean(axis=-1, keepdims=True)
                                 - zhat * (dzh * zhat).mean(axis=-1, keepdims=True))
    return {"dz": _frame(rb(dz), node), "dgamma": dgamma, "dbeta": dbeta, "dW": dW, "dwb": dwb, "dWo": dWo,
            "out": f["out"]}
