"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

# North-star gate: relative RMSE of every output against the FP64 oracle.
RMSE_REL_TOL = 2e-3


def rmse_rel(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.mean(ref * ref))
    num = np.sqrt(np.mean((x - ref) ** 2))
    return float(num / den) if den > 0 else float(num)


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


def check_lse(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    ninf = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), ninf), f"{what}: -inf pattern of LSE differs"
    fin = ~ninf
    if fin.any():
        err = np.max(np.abs(got[fin] - want[fin]) / (1.0 + np.abs(want[fin])))
        assert err < 5e-5, f"{what}: LSE max rel err {err}"
