"""Pins of the triangle-attention block oracle (oracle/trimodule.py) against things other than
itself.

- float64 torch autograd of the block written independently here (torch's layer_norm, an explicit
  softmax attention over einsum scores, and for the ending node attention along the columns of
  the untransposed tensor instead of a transpose): the output and all six gradients;
- central finite differences of sum(dout * out) along random directions, for every input;
- the LayerNorm output has zero mean and unit variance per position (gamma = 1, beta = 0);
- a closed form: with the q, k and gate rows of W and the bias weights zero, every unmasked key
  gets the same weight and the gate is 1/2, so out = (mean of v over the unmasked keys) Wo^T / 2;
- the BF16 storage rounding is the nearest BF16 value (ties to even).
"""
import numpy as np
import pytest
import torch

from bwd_tri_attn_gb300 import workloads as wl
from oracle import trimodule as om

EPS = 1e-5


def _inputs(B, N, c, H, d, seed, mask=("none",)):
    return wl.make_module_inputs(B, N, c, H, d, seed, mask)


def _torch_block(z, gamma, beta, W, wb, Wo, mask, H, d, node):
    """The block in float64 torch, with no transposed copy for the ending node."""
    B, N, _, c = z.shape
    hd = H * d
    zt = torch.nn.functional.layer_norm(z, (c,), gamma, beta, EPS)
    proj = zt @ W.T
    q, k, v, gl = (proj[..., s * hd:(s + 1) * hd].reshape(B, N, N, H, d) for s in range(4))
    bp = torch.einsum("bxyc,hc->bhxy", zt, wb)  # bias from pair position (x, y)
    m = torch.zeros(B, N, N, dtype=z.dtype) if mask is None else mask
    if node == 0:
        # slice i = first pair axis; query j, key k along the second
        s = torch.einsum("bijhd,bikhd->bhijk", q, k) / d ** 0.5 + bp[:, :, None, :, :] + m[:, None, :, None, :]
        p = torch.softmax(s, dim=-1)
        o = torch.einsum("bhijk,bikhd->bijhd", p, v)
    else:
        # slice i = second pair axis; query j, key k along the first; the bias of (j, k) comes
        # from pair position (k, j)
        s = (torch.einsum("bjihd,bkihd->bhijk", q, k) / d ** 0.5 + bp.transpose(2, 3)[:, :, None, :, :]
             + m[:, None, :, None, :])
        p = torch.softmax(s, dim=-1)
        o = torch.einsum("bhijk,bkihd->bjihd", p, v)
    go = torch.sigmoid(gl.reshape(B, N, N, hd)) * o.reshape(B, N, N, hd)
    return go @ Wo.T


@pytest.mark.parametrize("node,mask", [(0, ("none",)), (0, ("tail", 2)), (1, ("random", 0.3))])
def test_matches_torch_autograd(node, mask):
    H, d = 2, 4
    x = _inputs(2, 6, 8, H, d, seed=30 + node, mask=mask)
    args = [x[k] for k in ("z", "gamma", "beta", "W", "wb", "Wo")]
    g = om.bwd(*args, x["mask"], x["dout"], H, d, node=node)
    t = [a.double().clone().requires_grad_(True) for a in args]
    mk = None if x["mask"] is None else x["mask"].double()
    out = _torch_block(*t, mk, H, d, node)
    np.testing.assert_allclose(g["out"], out.detach().numpy(), rtol=1e-10, atol=1e-12)
    (out * x["dout"].double()).sum().backward()
    for name, tt in zip(("dz", "dgamma", "dbeta", "dW", "dwb", "dWo"), t):
        np.testing.assert_allclose(g[name], tt.grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=name)


@pytest.mark.parametrize("node", [0, 1])
def test_gradients_central_finite_differences(node):
    H, d = 2, 3
    x = _inputs(1, 4, 6, H, d, seed=40 + node, mask=("tail", 1))
    names = ("z", "gamma", "beta", "W", "wb", "Wo")
    base = {k: x[k].double().numpy() for k in names}
    dout = x["dout"].double().numpy()
    g = om.bwd(*[base[k] for k in names], x["mask"], dout, H, d, node=node)

    def loss(vals):
        return float(np.sum(dout * om.fwd(*[vals[k] for k in names], x["mask"], H, d, node=node)["out"]))

    rng = np.random.default_rng(50 + node)
    h = 1e-6
    for name, gname in zip(names, ("dz", "dgamma", "dbeta", "dW", "dwb", "dWo")):
        for _ in range(3):
            u = rng.standard_normal(base[name].shape)
            up, dn = dict(base), dict(base)
            up[name] = base[name] + h * u
            dn[name] = base[name] - h * u
            fd = (loss(up) - loss(dn)) / (2 * h)
            an = float(np.sum(g[gname] * u))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), f"{gname}: fd {fd} vs {an}"


def test_layer_norm_standardises():
    z = np.random.default_rng(60).standard_normal((2, 5, 5, 16)) * 3.0 + 1.5
    zt, mu, rstd = om.layer_norm(z, np.ones(16), np.zeros(16), EPS)
    np.testing.assert_allclose(zt.mean(axis=-1), 0.0, atol=1e-12)
    var = ((z - z.mean(axis=-1, keepdims=True)) ** 2).mean(axis=-1)
    np.testing.assert_allclose((zt ** 2).mean(axis=-1), var / (var + EPS), rtol=1e-12)
    np.testing.assert_allclose(mu, z.mean(axis=-1), rtol=1e-12)


@pytest.mark.parametrize("node", [0, 1])
def test_uniform_attention_closed_form(node):
    H, d, N, c = 2, 4, 7, 8
    x = _inputs(1, N, c, H, d, seed=70 + node, mask=("tail", 3))
    hd = H * d
    W = x["W"].double().numpy().copy()
    W[:2 * hd] = 0.0  # q and k rows: every score is the bias
    W[3 * hd:] = 0.0  # gate rows: sigmoid(0) = 1/2
    wb = np.zeros((H, c))
    z, gamma, beta, Wo = (x[k].double().numpy() for k in ("z", "gamma", "beta", "Wo"))
    out = om.fwd(z, gamma, beta, W, wb, Wo, x["mask"], H, d, node=node)["out"]
    zf = z if node == 0 else np.swapaxes(z, 1, 2)
    zt, _, _ = om.layer_norm(zf, gamma, beta, EPS)
    v = zt @ W[2 * hd:3 * hd].T                      # [B, slice, key, hd]
    vbar = v[:, :, :N - 3, :].mean(axis=2)           # mean over the unmasked keys of each slice
    ref = 0.5 * np.broadcast_to(vbar[:, :, None, :], v.shape) @ Wo.T
    if node == 1:
        ref = np.swapaxes(ref, 1, 2)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_bf16_rounding_is_nearest_even():
    # values exactly between two BF16 neighbours round to the one with an even last bit
    one_ulp = 2.0 ** -7
    x = np.array([1.0 + 0.5 * one_ulp, 1.0 + 1.5 * one_ulp, -(1.0 + 0.5 * one_ulp), 1.0 + 0.51 * one_ulp])
    np.testing.assert_array_equal(om.round_bf16(x), [1.0, 1.0 + 2 * one_ulp, -1.0, 1.0 + one_ulp])
    # and the result is a BF16 number: the low 16 bits of its FP32 pattern are zero
    y = om.round_bf16(np.random.default_rng(80).standard_normal(1000) * 100)
    assert np.all(y.astype(np.float32).view(np.uint32) & 0xFFFF == 0)
