"""GPU parity of the triangle-attention block (include/tri_module.h) against the FP64 oracle
(oracle/trimodule.py), through the C ABI.

Tolerances, from the arithmetic. The block stores about twenty BF16 tensors between its steps
(zt, q, k, v, gl, bias, O, go, out; dO, dgl, dq, dk, dv, dbias, dz), each rounding adding about
2^-9 / sqrt(3) relative error, which the following products carry on. The oracle run with the
same BF16 roundings (bf16=True) against the exact one measures that floor: 2.3e-3 to 5.6e-3
relative RMSE per output on the test shapes. The GPU path keeps the same roundings, and adds the
attention kernels' own error (within 2e-3 of their outputs, their gate) and FP32 accumulation.
So each output must be
  - within 1.2 * sqrt(floor^2 + (2e-3)^2) of the exact oracle (relative RMSE), and
  - within 3e-3 of the oracle with the same roundings.
The weight gradients are sums over every pair position in a fixed order: two calls must agree
to the bit.
"""
import numpy as np
import pytest
import torch

from bwd_tri_attn_gb300 import binding as tb
from bwd_tri_attn_gb300 import workloads as wl
from oracle import trimodule as om

pytestmark = pytest.mark.gpu

OUTS = ("out", "dz", "dgamma", "dbeta", "dW", "dwb", "dWo")
KEYS = ("z", "gamma", "beta", "W", "wb", "Wo")


def _rel(a, b):
    return float(np.sqrt(np.mean((a - b) ** 2)) / np.sqrt(np.mean(b ** 2)))


def _run_cuda(x, H, d, node):
    dev = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    args = [dev[k] for k in KEYS]
    out, saved = tb.module_forward(*args, dev["mask"], H, d, node=node)
    grads = tb.module_backward(*args, dev["mask"], saved, dev["dout"], H, d, node=node)
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
    return {k: t.detach().float().cpu().double().numpy() for k, t in zip(OUTS, (out,) + tuple(grads))}


def _oracle(x, H, d, node, bf16):
    g = om.bwd(*[x[k] for k in KEYS], x["mask"], x["dout"], H, d, node=node, bf16=bf16)
    return {k: g[k] for k in OUTS}


def _check(got, exact, mirrored):
    for k in OUTS:
        floor = _rel(mirrored[k], exact[k])
        e_ex, e_mi = _rel(got[k], exact[k]), _rel(got[k], mirrored[k])
        gate = 1.2 * np.sqrt(floor ** 2 + 2e-3 ** 2)
        assert np.all(np.isfinite(got[k])), k
        assert e_ex <= gate, f"{k}: {e_ex:.3e} from the exact oracle > {gate:.3e} (floor {floor:.3e})"
        assert e_mi <= 3e-3, f"{k}: {e_mi:.3e} from the oracle with the same BF16 roundings"


@pytest.mark.parametrize("w", [wl.MOD_TINY, wl.MOD_RAGGED, wl.MOD_ENDING], ids=lambda w: w.name)
def test_block_matches_oracle(w):
    x = wl.module_inputs_for(w)
    got = _run_cuda(x, w.H, w.d, w.node)
    _check(got, _oracle(x, w.H, w.d, w.node, False), _oracle(x, w.H, w.d, w.node, True))


@pytest.mark.parametrize("c,H,d,node", [(64, 4, 16, 0), (256, 2, 32, 1), (128, 8, 16, 0), (256, 8, 32, 0),
                                         (128, 6, 32, 1)])
def test_channel_and_head_variants(c, H, d, node):
    """Every LayerNorm width, H d from 64 to 256, both nodes, on a ragged N; H d = 192 puts the
    boundaries of the projections' four tensors inside GEMM tiles and between operand boxes."""
    x = wl.make_module_inputs(1, 40, c, H, d, seed=100 + c + H, mask=("tail", 3))
    got = _run_cuda(x, H, d, node)
    _check(got, _oracle(x, H, d, node, False), _oracle(x, H, d, node, True))


@pytest.mark.parametrize("B,N,node", [(1, 37, 0), (2, 21, 1), (3, 16, 0)])
def test_odd_and_batched_shapes(B, N, node):
    """N not a multiple of 8 (the attention's per-thread bias staging, positions not a multiple of
    the GEMM and store tiles), several batches on either node, the smallest N."""
    x = wl.make_module_inputs(B, N, 128, 4, 32, seed=200 + N, mask=("random", 0.2))
    got = _run_cuda(x, 4, 32, node)
    _check(got, _oracle(x, 4, 32, node, False), _oracle(x, 4, 32, node, True))


def test_magnitudes():
    """Output gradients at 2^-20 (the attention's operand scaling and the block's FP32 sums at tiny
    magnitudes), a common offset of 64 in z (the LayerNorm's centring), W and Wo times 2, and
    LayerNorm eps 1e-3."""
    x = wl.make_module_inputs(1, 48, 128, 4, 32, seed=300, mask=("tail", 4))
    x["dout"] = (x["dout"].float() * 2.0 ** -20).bfloat16()
    x["z"] = (x["z"].float() + 64.0).bfloat16()
    x["W"] = (x["W"].float() * 2.0).bfloat16()
    x["Wo"] = (x["Wo"].float() * 2.0).bfloat16()
    dev = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    args = [dev[k] for k in KEYS]
    out, saved = tb.module_forward(*args, dev["mask"], 4, 32, eps=1e-3)
    grads = tb.module_backward(*args, dev["mask"], saved, dev["dout"], 4, 32, eps=1e-3)
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
    got = {k: t.detach().float().cpu().double().numpy() for k, t in zip(OUTS, (out,) + tuple(grads))}
    ex = om.bwd(*[x[k] for k in KEYS], x["mask"], x["dout"], 4, 32, eps=1e-3)
    mi = om.bwd(*[x[k] for k in KEYS], x["mask"], x["dout"], 4, 32, eps=1e-3, bf16=True)
    _check(got, {k: ex[k] for k in OUTS}, {k: mi[k] for k in OUTS})


def test_crop384_full_oracle():
    w = wl.MOD_CROP384
    x = wl.module_inputs_for(w)
    got = _run_cuda(x, w.H, w.d, w.node)
    _check(got, _oracle(x, w.H, w.d, w.node, False), _oracle(x, w.H, w.d, w.node, True))


def test_crop768_full_oracle():
    """The benchmark's workload and launch configuration (crop 768, 48 masked keys), every output
    against the full oracle (about a minute of host time per oracle run)."""
    w = wl.MOD_CROP768
    x = wl.module_inputs_for(w)
    got = _run_cuda(x, w.H, w.d, w.node)
    _check(got, _oracle(x, w.H, w.d, w.node, False), _oracle(x, w.H, w.d, w.node, True))


def test_deterministic_across_calls():
    w = wl.MOD_RAGGED
    x = wl.module_inputs_for(w)
    a = _run_cuda(x, w.H, w.d, w.node)
    b = _run_cuda(x, w.H, w.d, w.node)
    for k in OUTS:
        assert np.array_equal(a[k], b[k]), k


def test_ending_node_is_starting_node_of_transposed_input():
    """The ending node on z equals the starting node on z with its pair axes swapped, the output
    and dz swapped back, with the mask unchanged (it is indexed by slice and key in both)."""
    w = wl.MOD_ENDING
    x = wl.module_inputs_for(w)
    end = _run_cuda(x, w.H, w.d, 1)
    xt = dict(x)
    xt["z"] = x["z"].transpose(1, 2).contiguous()
    xt["dout"] = x["dout"].transpose(1, 2).contiguous()
    start = _run_cuda(xt, w.H, w.d, 0)
    for k in ("out", "dz"):
        np.testing.assert_array_equal(end[k], np.swapaxes(start[k], 1, 2))
    for k in ("dgamma", "dbeta", "dW", "dwb", "dWo"):
        # the same sums over the same positions, visited in another order
        assert _rel(end[k], start[k]) <= 1e-5, k


def test_errors_before_launch():
    w = wl.MOD_TINY
    x = {k: (None if v is None else v.cuda()) for k, v in wl.module_inputs_for(w).items()}
    args = [x[k] for k in KEYS]
    shape = tb.module_shape_of(x["z"], w.H, w.d)
    small = torch.empty(tb.tri_module_saved_size(shape) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tb.TriAttnError) as e:
        tb.tri_module_fwd(shape, *args, x["mask"], torch.empty_like(x["z"]), small)
    assert e.value.code == -3
    out, saved = tb.module_forward(*args, x["mask"], w.H, w.d)
    ws = torch.empty(tb.tri_module_bwd_workspace_size(shape) - 256, dtype=torch.uint8, device="cuda")
    outs = tb.module_backward(*args, x["mask"], saved, x["dout"], w.H, w.d)
    with pytest.raises(tb.TriAttnError) as e:
        tb.tri_module_bwd(shape, *args, x["mask"], saved, x["dout"], *[torch.empty_like(o) for o in outs], ws)
    assert e.value.code == -3
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
