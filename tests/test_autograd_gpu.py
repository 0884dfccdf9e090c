"""The autograd glue (bwd_tri_attn_gb300/autograd.py) gives exactly the results of the direct C-ABI
calls it wraps: the same kernels with the same inputs, so every gradient must agree bit for bit.
"""
import pytest
import torch

from bwd_tri_attn_gb300 import autograd as ag
from bwd_tri_attn_gb300 import binding as tb
from bwd_tri_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _eq(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("node", [0, 1])
def test_attention_function_matches_direct_calls(node):
    x = {k: (None if v is None else v.cuda()) for k, v in
         wl.make_inputs(B=1, S=24, N=136, H=2, d=32, seed=70 + node, mask=("tail", 9)).items()}
    if node:
        x = {k: (v.transpose(1, 2).contiguous() if k in ("Q", "K", "V", "dO") else v) for k, v in x.items()}
    leaves = {k: x[k].clone().requires_grad_(True) for k in ("Q", "K", "V", "bias")}
    O = ag.triangle_attention(leaves["Q"], leaves["K"], leaves["V"], leaves["bias"], x["mask"], node=node)
    O.backward(x["dO"])
    O2, LSE, Ores = tb.forward(x["Q"], x["K"], x["V"], x["bias"], x["mask"], node=node)
    g = tb.backward(x["Q"], x["K"], x["V"], x["bias"], x["mask"], O2, Ores, LSE, x["dO"], node=node)
    torch.cuda.synchronize()
    assert _eq(O.detach(), O2)
    for name, ref in zip(("Q", "K", "V", "bias"), g):
        assert _eq(leaves[name].grad, ref), name
    assert tb.tri_attn_device_status() == 0


def test_block_module_matches_direct_calls():
    torch.manual_seed(0)
    m = ag.TriangleAttentionBlock(c=128, H=4, d=32, device="cuda")
    x = wl.make_module_inputs(1, 40, 128, 4, 32, seed=80, mask=("tail", 3))
    z = x["z"].cuda().requires_grad_(True)
    mask, dout = x["mask"].cuda(), x["dout"].cuda()
    out = m(z, mask)
    out.backward(dout)
    # the same call made directly, with the BF16 rounding of the FP32 master weights
    W, wb, Wo = (p.detach().to(torch.bfloat16) for p in (m.W, m.wb, m.Wo))
    g32, b32 = m.gamma.detach(), m.beta.detach()
    out2, saved = tb.module_forward(z.detach(), g32, b32, W, wb, Wo, mask, 4, 32)
    grads = tb.module_backward(z.detach(), g32, b32, W, wb, Wo, mask, saved, dout, 4, 32)
    torch.cuda.synchronize()
    assert _eq(out.detach(), out2)
    assert _eq(z.grad, grads[0])
    for p, ref in zip((m.gamma, m.beta, m.W, m.wb, m.Wo), grads[1:]):
        assert p.grad.dtype == torch.float32 and _eq(p.grad, ref)
    assert tb.tri_attn_device_status() == 0


@pytest.mark.parametrize("incoming,layout", [(False, 0), (True, 1)])
def test_multiplication_function_matches_direct_calls(incoming, layout):
    m = {k: v.cuda() for k, v in wl.make_mul_inputs(1, 72, 24, seed=90).items()}
    if layout == tb.LAYOUT_CHANNEL_MAJOR:
        m = {k: (v.permute(0, 3, 1, 2).contiguous() if k != "dX" else v) for k, v in m.items()}
    leaves = {k: m[k].clone().requires_grad_(True) for k in ("Pa", "Ga", "Pb", "Gb")}
    X = ag.triangle_multiplication(leaves["Pa"], leaves["Ga"], leaves["Pb"], leaves["Gb"], incoming, layout)
    X.backward(m["dX"])
    X2, A, Bm = tb.mul_forward(m["Pa"], m["Ga"], m["Pb"], m["Gb"], incoming=incoming, layout=layout)
    g = tb.mul_backward(m["Pa"], m["Ga"], m["Pb"], m["Gb"], A, Bm, m["dX"], incoming=incoming, layout=layout)
    torch.cuda.synchronize()
    assert _eq(X.detach(), X2)
    for name, ref in zip(("Pa", "Ga", "Pb", "Gb"), g):
        assert _eq(leaves[name].grad, ref), name
    assert tb.tri_attn_device_status() == 0


def test_second_derivative_is_refused():
    x = {k: (None if v is None else v.cuda()) for k, v in
         wl.make_inputs(B=1, S=16, N=40, H=1, d=16, seed=95).items()}
    q = x["Q"].clone().requires_grad_(True)
    O = ag.triangle_attention(q, x["K"], x["V"], x["bias"], None)
    (gq,) = torch.autograd.grad(O, q, x["dO"], create_graph=True)
    with pytest.raises(RuntimeError):
        gq.float().sum().backward()
    assert tb.tri_attn_device_status() == 0


def test_strided_inputs_give_the_contiguous_results():
    x = {k: (None if v is None else v.cuda()) for k, v in
         wl.make_inputs(B=1, S=20, N=72, H=2, d=32, seed=96, mask=("tail", 5)).items()}
    # the same values held transposed in memory: a strided view of a [B, N, S, H, d] tensor
    Qt = x["Q"].transpose(1, 2).contiguous().transpose(1, 2)
    assert not Qt.is_contiguous() and torch.equal(Qt, x["Q"])
    a = Qt.detach().requires_grad_(True)
    b = x["Q"].clone().requires_grad_(True)
    Oa = ag.triangle_attention(a, x["K"], x["V"], x["bias"], x["mask"])
    Ob = ag.triangle_attention(b, x["K"], x["V"], x["bias"], x["mask"])
    Oa.backward(x["dO"])
    Ob.backward(x["dO"])
    torch.cuda.synchronize()
    assert _eq(Oa.detach(), Ob.detach()) and _eq(a.grad, b.grad)
    assert tb.tri_attn_device_status() == 0
