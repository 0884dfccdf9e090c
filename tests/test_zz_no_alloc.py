"""The allocation-free backward entry point, tri_attn_bwd_static.

It serves callers that may not allocate device memory when they run the
backward pass (a plugin given only its input and output tensors, a service on a
fixed pre-planned memory budget): its scratch lives in one device array that
the library defines at file scope. These tests call it through the C ABI:

- where its work split equals tri_attn_bwd's, two calls in a row return exactly
  what tri_attn_bwd (caller-provided workspace) returns, bit for bit;
- at crop 768 the array cannot hold the dBias partial slots of the full split,
  so the entry point spreads the work over fewer clusters: dQ, dK and dV (whose
  reduction orders do not depend on the split) are still bitwise those of
  tri_attn_bwd, dBias (summed in another fixed order) matches the oracle and
  tri_attn_bwd within the RMSE gate, and two calls agree bit for bit;
- a shape too large for the array is refused with its own error code before
  anything runs.

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from bwd_tri_attn_gb300 import workloads as wl
from tests.parity_util import RMSE_REL_TOL, boundary_slices, check_elementwise, f64, oracle_full, rmse_rel

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


def _static_twice(tb, shape, d, O, Ores, LSE):
    results = []
    for _ in range(2):
        outs = [torch.full_like(d["Q"], float("nan")) for _ in range(3)] + [torch.full_like(d["bias"], float("nan"))]
        tb.tri_attn_bwd_static(shape, d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, Ores, LSE, d["dO"], *outs)
        torch.cuda.synchronize()
        assert tb.tri_attn_device_status() == 0
        results.append([t.clone() for t in outs])
    return results


def _same_bits(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


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
    assert tb.tri_attn_bwd_split(shape, True) == tb.tri_attn_bwd_split(shape, False)  # the same split
    for call, outs in enumerate(_static_twice(tb, shape, d, O, Ores, LSE)):
        for name, got, ref in zip(("dQ", "dK", "dV", "dBias"), outs, want):
            assert _same_bits(got, ref), f"call {call}: {name} differs from tri_attn_bwd"


def test_static_scratch_reduced_split_crop768(tb):
    # B = 1, H = 4, S = N = 768: the static array holds two dBias partial slots per head next to
    # the other scratch, while the device's full split needs more, so fewer clusters are used
    import oracle

    w = wl.CROP768
    x = wl.inputs_for(w)
    d = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    shape = tb.shape_of(d["Q"])
    nc_full, k_full = tb.tri_attn_bwd_split(shape, False)
    nc_static, k_static = tb.tri_attn_bwd_split(shape, True)
    assert nc_static < nc_full and k_static <= 2 < k_full, (nc_full, k_full, nc_static, k_static)

    O, LSE, Ores = tb.forward(d["Q"], d["K"], d["V"], d["bias"], d["mask"])
    want = tb.backward(d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, Ores, LSE, d["dO"])
    first, second = _static_twice(tb, shape, d, O, Ores, LSE)
    for name, a, b in zip(("dQ", "dK", "dV", "dBias"), first, second):
        assert _same_bits(a, b), f"{name}: two calls differ"
    for name, got, ref in zip(("dQ", "dK", "dV"), first[:3], want[:3]):
        assert _same_bits(got, ref), f"{name} differs from tri_attn_bwd (its order does not depend on the split)"
    e = rmse_rel(f64(first[3]), f64(want[3]))
    assert e <= RMSE_REL_TOL, f"dBias differs from tri_attn_bwd's by relative RMSE {e}"

    # against the oracle: slices at the reduced split's cluster boundaries, dBias rows of every head
    sl, _ = boundary_slices(shape, w.slices, static_entry=True)
    sl = sorted(set(sl + [0, w.N - 1]))
    sub = {k: (v[:, sl] if (v is not None and k in ("Q", "K", "V", "dO", "mask")) else v) for k, v in x.items()}
    ref = oracle_full(sub)
    for name, got in zip(("dQ", "dK", "dV"), first[:3]):
        g = f64(got[:, sl].cpu())
        assert rmse_rel(g, ref[name]) <= RMSE_REL_TOL, name
        check_elementwise(g, ref[name], f"static crop768 {name}")
    rows = [(0, h, j) for h in range(w.H) for j in (0, 383, w.N - 1)]
    want_rows = oracle.dbias_rows(x["Q"], x["K"], x["V"], x["bias"], x["mask"], x["dO"], rows)
    got_rows = np.stack([f64(first[3][b, h, j].cpu()) for (b, h, j) in rows])
    assert rmse_rel(got_rows, want_rows) <= RMSE_REL_TOL
    check_elementwise(got_rows, want_rows, "static crop768 dBias rows")


def _static_need_bytes(B, S, N, H):
    """Bytes the static entry point needs at the least (one dBias partial slot per head): its
    scratch layout is D | scale exponents | transposed bias | partial slots, each 256-byte aligned."""
    def up(n):
        return (n + 255) // 256 * 256
    NP = (N + 127) // 128 * 128
    return up(4 * B * S * H * N) + up(16 * B * S * H) + up(2 * B * H * NP * NP) + 4 * B * H * NP * NP


def test_static_scratch_rejects_oversized_shape(tb):
    B, S, N, H, d = 1, 1024, 1024, 4, 32
    cap = 32 * 1024 * 1024  # TRI_ATTN_STATIC_WORKSPACE_BYTES
    # precondition, checked before the call: this shape really exceeds the array, so the call must
    # stop at its size check (and the tensors below are real, so even a call that went further would
    # touch only valid memory)
    assert _static_need_bytes(B, S, N, H) > cap
    shape = tb.Shape(B, S, N, H, d, d ** -0.5, tb.NODE_STARTING)
    dev = "cuda"
    pair = [torch.zeros((B, S, N, H, d), dtype=torch.bfloat16, device=dev) for _ in range(9)]
    Q, K, V, O, Ores, dO, dQ, dK, dV = pair
    bias = torch.zeros((B, H, N, N), dtype=torch.bfloat16, device=dev)
    dBias = torch.zeros_like(bias)
    LSE = torch.zeros((B, S, H, N), dtype=torch.float32, device=dev)
    with pytest.raises(tb.TriAttnError) as ei:
        tb.tri_attn_bwd_static(shape, Q, K, V, bias, None, O, Ores, LSE, dO, dQ, dK, dV, dBias)
    assert ei.value.code == -6
    assert "static workspace" in tb.strerror(ei.value.code)
    with pytest.raises(tb.TriAttnError) as ei:
        tb.tri_attn_bwd_split(shape, True)
    assert ei.value.code == -6
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
