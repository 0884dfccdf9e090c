"""Seeded synthetic inputs for triangle attention and the triangle multiplicative update.

This module holds no arithmetic of the method: it only draws random tensors
(CPU ``torch.Generator``, float32 normal draws rounded to BF16) in the shapes,
value distributions and padding patterns of the crop sizes that the
TurboPairFormer paper evaluates (arXiv 2610.05854v1, Abstract: BF16 inputs,
crops 384/640/768, head dims 16/32). Both the CUDA path's tests and the oracle
are fed from here.

Layouts: Q, K, V, dO [B,S,N,H,d] (S = number of row-slices, equal to N for a
square pair tensor); bias [B,H,N,N]; mask [B,S,N] additive BF16 (0 or -inf) or
None. Triangle multiplication: projections P_a, G_a, P_b, G_b [B,N,N,C] (pair
layout) and the output gradient dX [B,C,N,N] (channel-major), with the pair
channel count of AlphaFold3-style trunks (128) at the attention's crop sizes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    """One named input recipe."""

    name: str
    B: int
    N: int
    H: int
    d: int
    seed: int
    value_std: float = 1.0
    bias_std: float = 1.0
    # mask kinds: "none" (NULL mask), "zeros" (all valid but present),
    # ("tail", n) last n keys masked in every slice, ("random", frac) a random
    # fraction of keys masked per batch, shared by all slices.
    mask: tuple = ("none",)
    S: int | None = None  # number of slices; defaults to N
    notes: str = field(default="", compare=False)

    @property
    def slices(self) -> int:
        return self.N if self.S is None else self.S

    def flops(self) -> float:
        """Algorithmic fwd+bwd FLOPs: 4 (fwd) + 10 (bwd incl. one recompute) x B*S*H*N^2*d."""
        return 14.0 * self.B * self.slices * self.H * self.N * self.N * self.d


TINY = Workload("tiny_n32_h2_d16", B=1, N=32, H=2, d=16, seed=0, mask=("none",),
                notes="tiny starting-node case, no mask")
PAD128 = Workload("pad_n128_h4_d32", B=1, N=128, H=4, d=32, seed=1, value_std=0.5,
                  mask=("tail", 13), notes="last 13 keys padding-masked in every slice")
CROP384 = Workload("crop384_h4_d32", B=1, N=384, H=4, d=32, seed=2, bias_std=2.0,
                   mask=("zeros",), notes="all-valid mask tensor, bias sigma 2")
CROP640_D16 = Workload("crop640_h4_d16", B=1, N=640, H=4, d=16, seed=3,
                       mask=("random", 0.05), notes="5% random key mask per batch")
CROP640_D32 = Workload("crop640_h4_d32", B=1, N=640, H=4, d=32, seed=3,
                       mask=("random", 0.05), notes="5% random key mask per batch")
CROP768 = Workload("crop768_h4_d32", B=1, N=768, H=4, d=32, seed=4,
                   mask=("tail", 48), notes="last 48 keys padding-masked; headline size")

ALL = {w.name: w for w in (TINY, PAD128, CROP384, CROP640_D16, CROP640_D32, CROP768)}


def _normal(gen, shape, std):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def make_mask(kind, B, S, N, gen) -> torch.Tensor | None:
    """Additive BF16 key mask [B,S,N] for a mask recipe (see ``Workload.mask``)."""
    tag = kind[0]
    if tag == "none":
        return None
    m = torch.zeros((B, S, N), dtype=torch.float32)
    if tag == "zeros":
        pass
    elif tag == "tail":
        n = int(kind[1])
        if n > 0:
            m[:, :, N - n:] = float("-inf")
    elif tag == "random":
        n = int(round(float(kind[1]) * N))
        for b in range(B):
            keys = torch.randperm(N, generator=gen)[:n]
            m[b, :, keys] = float("-inf")
    elif tag == "slices":
        # every key of the listed slices is masked (fully masked rows)
        for i in kind[1]:
            m[:, int(i), :] = float("-inf")
    else:
        raise ValueError(f"unknown mask kind {kind!r}")
    return m.to(torch.bfloat16)


def make_inputs(B, S, N, H, d, seed, value_std=1.0, bias_std=1.0, mask=("none",)):
    """Draws Q, K, V, dO, bias and mask (CPU, BF16) for one seed.

    Draw order is fixed: Q, K, V, dO, bias, then the mask's own draws.
    """
    gen = torch.Generator().manual_seed(int(seed))
    shape = (B, S, N, H, d)
    Q = _normal(gen, shape, value_std)
    K = _normal(gen, shape, value_std)
    V = _normal(gen, shape, value_std)
    dO = _normal(gen, shape, value_std)
    bias = _normal(gen, (B, H, N, N), bias_std)
    m = make_mask(mask, B, S, N, gen)
    return {"Q": Q, "K": K, "V": V, "dO": dO, "bias": bias, "mask": m}


def inputs_for(w: Workload, slices: int | None = None):
    """Inputs of a named workload; ``slices`` overrides S (a bounded sample)."""
    S = w.slices if slices is None else int(slices)
    return make_inputs(w.B, S, w.N, w.H, w.d, w.seed, w.value_std, w.bias_std, w.mask)


def scale_pow2(x: dict, exps: dict) -> dict:
    """A copy of the inputs with the named tensors multiplied by 2**e (exact in BF16 while the
    results stay in BF16's normal range): the same problem at another magnitude."""
    out = dict(x)
    for k, e in exps.items():
        out[k] = (x[k].float() * (2.0 ** e)).to(torch.bfloat16)
    return out


def ending_node(t: torch.Tensor) -> torch.Tensor:
    """Transposes the pair axes (1 <-> 2) of a [B,S,N,...] tensor, contiguous copy.

    The ending-node variant of triangle attention is the same operation on the
    transposed pair tensor.
    """
    return t.transpose(1, 2).contiguous()


@dataclass(frozen=True)
class MulWorkload:
    """One named input recipe of the triangle multiplicative update."""

    name: str
    B: int
    N: int
    C: int
    seed: int
    std: float = 1.0       # projections P_a, P_b
    gate_std: float = 1.0  # gate logits G_a, G_b
    notes: str = field(default="", compare=False)

    def flops(self) -> float:
        """Algorithmic FLOPs of the contraction: 2 B C N^3 forward, twice that backward."""
        return 2.0 * self.B * self.C * float(self.N) ** 3


MUL_TINY = MulWorkload("mul_tiny_n16_c8", B=1, N=16, C=8, seed=10, notes="smallest supported shape")
MUL_RAGGED = MulWorkload("mul_ragged_b2_n72_c24", B=2, N=72, C=24, seed=11, notes="N and C off every tile size")
MUL_CROP384 = MulWorkload("mul_crop384_c128", B=1, N=384, C=128, seed=12, notes="crop 384, 128 pair channels")
MUL_CROP768 = MulWorkload("mul_crop768_c128", B=1, N=768, C=128, seed=13, notes="crop 768, 128 pair channels")

MUL_ALL = {w.name: w for w in (MUL_TINY, MUL_RAGGED, MUL_CROP384, MUL_CROP768)}


def make_mul_inputs(B, N, C, seed, std=1.0, gate_std=1.0):
    """Draws P_a, G_a, P_b, G_b ([B,N,N,C]) and dX ([B,C,N,N]) as BF16 on the CPU, in that order."""
    gen = torch.Generator().manual_seed(int(seed))
    pair = (B, N, N, C)
    return {"Pa": _normal(gen, pair, std), "Ga": _normal(gen, pair, gate_std), "Pb": _normal(gen, pair, std),
            "Gb": _normal(gen, pair, gate_std), "dX": _normal(gen, (B, C, N, N), 1.0)}


def mul_inputs_for(w: MulWorkload):
    return make_mul_inputs(w.B, w.N, w.C, w.seed, w.std, w.gate_std)


@dataclass(frozen=True)
class ModWorkload:
    """One named input recipe of the triangle-attention block (LayerNorm, projections, attention,
    gate, output projection) around the attention core."""

    name: str
    B: int
    N: int
    c: int   # pair channels
    H: int
    d: int
    seed: int
    mask: tuple = ("none",)
    node: int = 0
    notes: str = field(default="", compare=False)

    def flops(self) -> float:
        """Algorithmic fwd+bwd FLOPs: the attention's 14 B N^3 H d, plus the projections' GEMMs
        (2 M c (5 H d + H) forward, twice that backward, M = B N^2)."""
        m = float(self.B) * self.N * self.N
        hd = self.H * self.d
        return 14.0 * m * self.N * hd + 3 * 2.0 * m * self.c * (5 * hd + self.H)


MOD_TINY = ModWorkload("mod_tiny_n24_c64_h2_d32", B=1, N=24, c=64, H=2, d=32, seed=20, notes="smallest tile case")
MOD_RAGGED = ModWorkload("mod_ragged_b2_n72_c128_h4_d16", B=2, N=72, c=128, H=4, d=16, seed=21,
                         mask=("tail", 5), notes="N off every tile size, d = 16, tail mask")
MOD_ENDING = ModWorkload("mod_ending_n136_c128_h4_d32", B=1, N=136, c=128, H=4, d=32, seed=22,
                         mask=("random", 0.1), node=1, notes="ending node, ragged N, random key mask")
MOD_CROP384 = ModWorkload("mod_crop384_c128_h4_d32", B=1, N=384, c=128, H=4, d=32, seed=23, mask=("zeros",),
                          notes="crop 384 with AlphaFold3-style pair width 128")
MOD_CROP768 = ModWorkload("mod_crop768_c128_h4_d32", B=1, N=768, c=128, H=4, d=32, seed=24, mask=("tail", 48),
                          notes="crop 768, last 48 keys padding-masked")

MOD_ALL = {w.name: w for w in (MOD_TINY, MOD_RAGGED, MOD_ENDING, MOD_CROP384, MOD_CROP768)}


def make_module_inputs(B, N, c, H, d, seed, mask=("none",)):
    """Draws, in this order: z [B,N,N,c], dout [B,N,N,c] (BF16, unit normal), the LayerNorm scale
    and shift (FP32, 1 + 0.1 n and 0.1 n), the projection weights W [4 H d, c] and wb [H, c] (BF16,
    normal / sqrt(c)) and Wo [c, H d] (BF16, normal / sqrt(H d)), then the mask's own draws."""
    gen = torch.Generator().manual_seed(int(seed))
    hd = H * d
    z = _normal(gen, (B, N, N, c), 1.0)
    dout = _normal(gen, (B, N, N, c), 1.0)
    gamma = 1.0 + 0.1 * torch.randn((c,), generator=gen, dtype=torch.float32)
    beta = 0.1 * torch.randn((c,), generator=gen, dtype=torch.float32)
    W = _normal(gen, (4 * hd, c), c ** -0.5)
    wb = _normal(gen, (H, c), c ** -0.5)
    Wo = _normal(gen, (c, hd), hd ** -0.5)
    m = make_mask(mask, B, N, N, gen)
    return {"z": z, "dout": dout, "gamma": gamma, "beta": beta, "W": W, "wb": wb, "Wo": Wo, "mask": m}


def module_inputs_for(w: ModWorkload):
    return make_module_inputs(w.B, w.N, w.c, w.H, w.d, w.seed, w.mask)
