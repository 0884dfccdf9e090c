"""The allocation-free backward entry point, tri_attn_bwd_static.

It serves callers that may not allocate device memory when they run the
backward pass (a plugin given only its input and output tensors, a service on a
fixed pre-planned memory budget): its scratch lives in one device array that
the library defines at file scope. These tests call it through the C ABI and
check that two calls in a row give what tri_attn_bwd (caller-provided
workspace) gives, within the suite's RMSE tolerance, and that a shape too large
for the array is refused with its own error code before anything runs.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from bwd_tri_attn_gb300 import workloads as wl
from tests.parity_util import RMSE_REL_TOL, f64, rmse_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bwd_tri_attn_gb300 import _build
    from bwd_tri_attn_gb300 import binding
    _build.build()
    binding.load()
    return binding


@pytest.mark.parametrize("cfg", [
    dict(B=1, S=64, N=200, H=2, d=32, seed=31, mask=("random", 0.1)),
    dict(B=2, S=24, N=136, H=3, d=16, seed=32, mask=("tail", 9)),
])
def test_static_scratch_matches_workspace_entry_point(tb, cfg):
    x = wl.make_inputs(**cfg)
    d = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    O, LSE, Ores = tb.forward(d["Q"], d["K"], d["V"], d["bias"], d["mask"])
    want = tb.backward(d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, Ores, LSE, d["dO"])
    shape = tb.shape_of(d["Q"])
    for call in range(2):
        outs = [torch.full_like(d["Q"], float("nan")) for _ in range(3)] + [torch.full_like(d["bias"], float("nan"))]
        tb.tri_attn_bwd_static(shape, d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, Ores, LSE, d["dO"], *outs)
        torch.cuda.synchronize()
        assert tb.tri_attn_device_status() == 0
        for name, got, ref in zip(("dQ", "dK", "dV", "dBias"), outs, want):
            assert not torch.isnan(got.float()).any(), f"call {call}: {name} not fully written"
            e = rmse_rel(f64(got), f64(ref))
            assert e <= RMSE_REL_TOL, f"call {call}: {name} differs from tri_attn_bwd, relative RMSE {e}"


def test_static_scratch_rejects_oversized_shape(tb):
    lib = tb.load()
    shape = tb.Shape(1, 1024, 1024, 4, 32, 0.17677669)
    fake = [ctypes.c_void_p(0x10000)] * 13
    rc = lib.tri_attn_bwd_static(shape, *fake, None)
    assert rc == -6
    assert "static workspace" in tb.strerror(rc)
