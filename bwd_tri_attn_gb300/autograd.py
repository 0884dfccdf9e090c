"""PyTorch autograd glue over the C ABI (argument marshalling only).

Every forward and backward step runs in the library's kernels through ``binding``; these classes
only keep the tensors the backward pass needs and hand gradients back in the dtypes autograd
expects. There is no CPU path: the library raises if it is missing or a call fails. Inputs are
made contiguous (a no-op for contiguous tensors); dtypes and sizes are checked by the binding. The
backward passes are differentiable once (no second derivatives).

- ``triangle_attention(Q, K, V, bias, mask=None, node=NODE_STARTING)``: the attention core
  (include/tri_attn.h) with its residual-compensated backward; gradients for Q, K, V and bias.
- ``triangle_multiplication(Pa, Ga, Pb, Gb, incoming=False, layout=LAYOUT_PAIR)``: the triangle
  multiplicative update (include/tri_mul.h); X channel-major [B, C, N, N], gradients for the four
  projections in their layout.
- ``triangle_attention_block(z, gamma, beta, W, wb, Wo, mask, H, d, node, eps)`` and
  ``TriangleAttentionBlock``: the surrounding block (include/tri_module.h). The weights may be FP32
  masters: the forward uses their BF16 rounding (as mixed-precision training does) and the
  backward returns the library's FP32 weight gradients in the masters' dtype.
"""
from __future__ import annotations

import math

import torch
from torch.autograd.function import once_differentiable

from . import binding as tb


class _TriangleAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Q, K, V, bias, mask, node):
        Q, K, V, bias = (t.contiguous() for t in (Q, K, V, bias))
        mask = None if mask is None else mask.contiguous()
        O, LSE, Ores = tb.forward(Q, K, V, bias, mask, node=node)
        ctx.node = node
        ctx.save_for_backward(Q, K, V, bias, mask, O, Ores, LSE)
        return O

    @staticmethod
    @once_differentiable
    def backward(ctx, dO):
        Q, K, V, bias, mask, O, Ores, LSE = ctx.saved_tensors
        dQ, dK, dV, dBias = tb.backward(Q, K, V, bias, mask, O, Ores, LSE,
                                        dO.to(torch.bfloat16).contiguous(), node=ctx.node)
        return dQ, dK, dV, dBias, None, None


def triangle_attention(Q, K, V, bias, mask=None, node=tb.NODE_STARTING):
    """O of the attention core for BF16 CUDA tensors Q, K, V [B, S, N, H, d] (starting node; the
    ending node takes [B, N, S, H, d] in place), bias [B, H, N, N], mask [B, S, N] or None."""
    return _TriangleAttention.apply(Q, K, V, bias, mask, node)


class _TriangleMultiplication(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Pa, Ga, Pb, Gb, incoming, layout):
        Pa, Ga, Pb, Gb = (t.contiguous() for t in (Pa, Ga, Pb, Gb))
        X, A, Bm = tb.mul_forward(Pa, Ga, Pb, Gb, incoming=incoming, layout=layout)
        ctx.cfg = (incoming, layout)
        ctx.save_for_backward(Pa, Ga, Pb, Gb, A, Bm)
        return X

    @staticmethod
    @once_differentiable
    def backward(ctx, dX):
        Pa, Ga, Pb, Gb, A, Bm = ctx.saved_tensors
        incoming, layout = ctx.cfg
        grads = tb.mul_backward(Pa, Ga, Pb, Gb, A, Bm, dX.to(torch.bfloat16).contiguous(), incoming=incoming,
                                layout=layout)
        return (*grads, None, None)


def triangle_multiplication(Pa, Ga, Pb, Gb, incoming=False, layout=tb.LAYOUT_PAIR):
    """X [B, C, N, N] of the triangle multiplicative update for BF16 CUDA projections and gate
    logits (layout LAYOUT_PAIR: [B, N, N, C]; LAYOUT_CHANNEL_MAJOR: [B, C, N, N])."""
    return _TriangleMultiplication.apply(Pa, Ga, Pb, Gb, incoming, layout)


class _TriangleAttentionBlock(torch.autograd.Function):
    @staticmethod
    def forward(ctx, z, gamma, beta, W, wb, Wo, mask, H, d, node, eps):
        z = z.contiguous()
        mask = None if mask is None else mask.contiguous()
        bf = [t.to(torch.bfloat16).contiguous() for t in (W, wb, Wo)]
        g32, b32 = gamma.float().contiguous(), beta.float().contiguous()
        out, saved = tb.module_forward(z, g32, b32, *bf, mask, H, d, node=node, eps=eps)
        ctx.meta = (H, d, node, eps, [t.dtype for t in (gamma, beta, W, wb, Wo)])
        ctx.save_for_backward(z, g32, b32, *bf, mask, saved)
        return out

    @staticmethod
    @once_differentiable
    def backward(ctx, dout):
        z, g32, b32, W, wb, Wo, mask, saved = ctx.saved_tensors
        H, d, node, eps, dtypes = ctx.meta
        grads = tb.module_backward(z, g32, b32, W, wb, Wo, mask, saved, dout.to(torch.bfloat16).contiguous(),
                                   H, d, node=node, eps=eps)
        dz = grads[0]
        wgrads = [g.to(dt) for g, dt in zip(grads[1:], dtypes)]
        return (dz, *wgrads, None, None, None, None, None)


def triangle_attention_block(z, gamma, beta, W, wb, Wo, mask, H, d, node=tb.NODE_STARTING, eps=1e-5):
    """The triangle-attention block on the BF16 pair representation z [B, N, N, c]: LayerNorm
    (gamma, beta [c]), projections W [4 H d, c] (q, k, v, gate rows) and wb [H, c], the attention,
    the sigmoid gate and the output projection Wo [c, H d]."""
    return _TriangleAttentionBlock.apply(z, gamma, beta, W, wb, Wo, mask, H, d, node, eps)


class TriangleAttentionBlock(torch.nn.Module):
    """The triangle-attention block as a module with FP32 master parameters (initialised like the
    seeded test inputs: gamma 1, beta 0, W and wb normal / sqrt(c), Wo normal / sqrt(H d))."""

    def __init__(self, c: int = 128, H: int = 4, d: int = 32, node: int = tb.NODE_STARTING, eps: float = 1e-5,
                 device=None):
        super().__init__()
        self.c, self.H, self.d, self.node, self.eps = c, H, d, node, eps
        f32 = dict(dtype=torch.float32, device=device)
        self.gamma = torch.nn.Parameter(torch.ones(c, **f32))
        self.beta = torch.nn.Parameter(torch.zeros(c, **f32))
        self.W = torch.nn.Parameter(torch.randn(4 * H * d, c, **f32) / math.sqrt(c))
        self.wb = torch.nn.Parameter(torch.randn(H, c, **f32) / math.sqrt(c))
        self.Wo = torch.nn.Parameter(torch.randn(c, H * d, **f32) / math.sqrt(H * d))

    def forward(self, z, mask=None):
        return triangle_attention_block(z, self.gamma, self.beta, self.W, self.wb, self.Wo, mask, self.H, self.d,
                                        self.node, self.eps)
