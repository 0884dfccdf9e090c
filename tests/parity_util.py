"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle, compare."""
from __future__ import annotations

import os

import numpy as np
import torch

# North-star gate: relative RMSE of every output against the FP64 oracle.
RMSE_REL_TOL = 2e-3

# Per-element gate, beside the whole-tensor RMSE (which one wrong store barely moves):
#   |x - ref| <= ELEM_ULPS * ulp_bf16(ref) + ELEM_EPS * rms(ref)
# The first term covers the BF16 rounding of the result (half an ulp) plus relative errors of the
# same size; the second covers the absolute error the FP32/FP16 arithmetic accumulates in a sum
# whose terms cancel (a few times the 1e-3 relative RMSE, at the tail of millions of elements).
# A wrong 32-byte store moves most of its 16 elements by about rms(ref) and fails it.
ELEM_ULPS = 1.0
ELEM_EPS = 2e-2


def rmse_rel(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.mean(ref * ref))
    num = np.sqrt(np.mean((x - ref) ** 2))
    return float(num / den) if den > 0 else float(num)


def ulp_bf16(ref) -> np.ndarray:
    """Spacing of BF16 numbers at |ref| (8 significant bits)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def elementwise_excess(x, ref, ulps=ELEM_ULPS) -> float:
    """Largest (|x - ref| - ulps * ulp_bf16(ref)) / rms(ref) over all elements: the smallest ELEM_EPS
    the element-wise gate would need."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    if rms == 0:
        return float(np.max(np.abs(x))) if x.size else 0.0
    return float(np.max((np.abs(x - ref) - ulps * ulp_bf16(ref)) / rms))


def check_elementwise(x, ref, what=""):
    e = elementwise_excess(x, ref)
    log = os.environ.get("TRI_ATTN_ELEM_LOG")
    if log:
        with open(log, "a") as f:
            f.write(f"{what}\t{e:.6g}\n")
    assert e <= ELEM_EPS, f"{what}: an element is {e:.3g} rms(ref) beyond its BF16 ulp (gate {ELEM_EPS})"
    return e


def f64(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def to_device(x: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device).contiguous()) for k, v in x.items()}


PAIR = ("Q", "K", "V", "dO", "O", "Ores", "dQ", "dK", "dV")  # tensors laid out as pair tensors


def run_cuda(x: dict, residual=True, scale=None, workspace=None, node=0):
    """One forward + backward through the C ABI; returns CPU tensors.

    ``x`` is in the attention's own terms ([B, S, N, H, d] activations). With node = 1 the
    activations are handed to the library as ending-node pair tensors ([B, N, S, H, d], slices
    along the second pair axis) and its outputs are mapped back, so results compare directly.
    """
    from bwd_tri_attn_gb300 import binding as tb

    dx = to_device(x)
    if node:
        dx = {k: (v.transpose(1, 2).contiguous() if k in PAIR else v) for k, v in dx.items()}
    O, LSE, Ores = tb.forward(dx["Q"], dx["K"], dx["V"], dx["bias"], dx["mask"], scale=scale, residual=True,
                              node=node)
    dQ, dK, dV, dBias = tb.backward(dx["Q"], dx["K"], dx["V"], dx["bias"], dx["mask"], O,
                                    Ores if residual else None, LSE, dx["dO"], scale=scale,
                                    workspace=workspace, node=node)
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
    out = dict(O=O, LSE=LSE, Ores=Ores, dQ=dQ, dK=dK, dV=dV, dBias=dBias)
    if node:
        out = {k: (v.transpose(1, 2) if k in PAIR else v) for k, v in out.items()}
    return {k: v.contiguous().cpu() for k, v in out.items()}


def oracle_full(x: dict, scale=None):
    import oracle

    O, LSE = oracle.fwd(x["Q"], x["K"], x["V"], x["bias"], x["mask"], scale)
    g = oracle.bwd(x["Q"], x["K"], x["V"], x["bias"], x["mask"], x["dO"], scale)
    return dict(O=O, LSE=LSE, **g)


def boundary_slices(shape, S, static_entry=False):
    """Slices that straddle the backward's cluster-range boundaries (for every boundary, the last
    (head, slice) pair of one cluster and the first of the next), from the split the library reports."""
    from bwd_tri_attn_gb300 import binding as tb

    nc, _ = tb.tri_attn_bwd_split(shape, static_entry)
    w = shape.B * shape.H * S
    out = set()
    for c in range(1, nc):
        x = c * w // nc
        out.update({(x - 1) % S, x % S})
    return sorted(out), nc


def check_lse(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    ninf = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern of LSE differs"
    fin = ~ninf
    if fin.any():
        err = np.max(np.abs(got[fin] - want[fin]) / (1.0 + np.abs(want[fin])))
        assert err < 5e-5, f"{what}: LSE max rel err {err}"
