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


def run_cuda(x: dict, residual=True, scale=None, workspace=None):
    """One forward + backward through the C ABI; returns CPU tensors."""
    from bwd_tri_attn_gb300 import binding as tb

    dx = to_device(x)
    O, LSE, Ores = tb.forward(dx["Q"], dx["K"], dx["V"], dx["bias"], dx["mask"], scale=scale, residual=True)
    dQ, dK, dV, dBias = tb.backward(dx["Q"], dx["K"], dx["V"], dx["bias"], dx["mask"], O,
                                    Ores if residual else None, LSE, dx["dO"], scale=scale,
                                    workspace=workspace)
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
    out = dict(O=O, LSE=LSE, Ores=Ores, dQ=dQ, dK=dK, dV=dV, dBias=dBias)
    return {k: v.cpu() for k, v in out.items()}


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
