"""Pins of the triangle-multiplication oracle (oracle/trimul.py) against things other than itself.

- explicit triple loops on tiny inputs (not einsum) for both directions;
- the incoming update is the outgoing update of the pair-transposed operands;
- with a = b the outgoing update is symmetric in (i, j);
- sigmoid(0) = 1/2 halves P exactly, so X(G = 0) = X of P alone / 4;
- per channel, X is the matrix product of the channel's N x N operand slices (numpy matmul);
- central finite differences and float64 torch autograd of sum(dX * X) for all four gradients
  (BF16 storage of the gated operands switched off, as a derivative through rounding is meaningless).
"""
import itertools

import numpy as np
import pytest
import torch

from oracle import trimul as om


def _draw(B, N, C, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return [g.standard_normal((B, N, N, C)) * scale for _ in range(4)]


def _loops(a, b, incoming):
    B, N, _, C = a.shape
    X = np.zeros_like(a)
    for bb, i, j, c in itertools.product(range(B), range(N), range(N), range(C)):
        s = 0.0
        for k in range(N):
            s += a[bb, k, i, c] * b[bb, k, j, c] if incoming else a[bb, i, k, c] * b[bb, j, k, c]
        X[bb, i, j, c] = s
    return X


@pytest.mark.parametrize("incoming", [False, True])
def test_contraction_matches_explicit_loops(incoming):
    pa, ga, pb, gb = _draw(2, 5, 3, seed=1)
    a, b = om.gated(pa, ga), om.gated(pb, gb)
    np.testing.assert_allclose(om.fwd(pa, ga, pb, gb, incoming), _loops(a, b, incoming), rtol=1e-12, atol=1e-12)


def test_gating_is_sigmoid_times_projection_stored_in_bf16():
    pa, ga, _, _ = _draw(1, 4, 2, seed=2)
    a = om.gated(pa, ga)
    exact = pa / (1.0 + np.exp(-ga))
    # BF16 keeps 8 significant bits: round to nearest is within half an ulp (2^-8 relative)
    assert np.all(np.abs(a - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-300)
    # and the stored values are BF16 numbers: the low 16 bits of their FP32 patterns are zero
    bits = a.astype(np.float32).view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)


def test_incoming_is_outgoing_of_transposed_operands():
    pa, ga, pb, gb = _draw(2, 7, 4, seed=3)
    t = lambda x: np.ascontiguousarray(np.swapaxes(x, 1, 2))
    np.testing.assert_allclose(om.fwd(pa, ga, pb, gb, incoming=True), om.fwd(t(pa), t(ga), t(pb), t(gb), incoming=False),
                               rtol=1e-13, atol=1e-13)


def test_outgoing_symmetric_when_operands_equal():
    pa, ga, _, _ = _draw(1, 9, 3, seed=4)
    X = om.fwd(pa, ga, pa, ga)
    np.testing.assert_allclose(X, np.swapaxes(X, 1, 2), rtol=1e-13, atol=1e-13)


def test_zero_gate_halves_the_projections():
    pa, _, pb, _ = _draw(1, 6, 2, seed=5)
    pa, pb = om.round_bf16(pa), om.round_bf16(pb)  # BF16 inputs: halving them is exact in BF16
    z = np.zeros_like(pa)
    np.testing.assert_allclose(om.fwd(pa, z, pb, z), 0.25 * _loops(pa, pb, False), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("incoming", [False, True])
def test_channel_slices_are_matrix_products(incoming):
    pa, ga, pb, gb = _draw(2, 8, 3, seed=6)
    a, b = om.gated(pa, ga), om.gated(pb, gb)
    X = om.fwd(pa, ga, pb, gb, incoming)
    for bb in range(2):
        for c in range(3):
            A, Bm = a[bb, :, :, c], b[bb, :, :, c]
            ref = A.T @ Bm if incoming else A @ Bm.T
            np.testing.assert_allclose(X[bb, :, :, c], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("incoming", [False, True])
def test_gradients_central_finite_differences(incoming):
    pa, ga, pb, gb = _draw(1, 4, 2, seed=7)
    dX = np.random.default_rng(8).standard_normal(pa.shape)
    grads = om.bwd(pa, ga, pb, gb, dX, incoming, bf16=False)
    args = [pa, ga, pb, gb]
    h = 1e-6
    for n, name in enumerate(("dPa", "dGa", "dPb", "dGb")):
        fd = np.zeros_like(pa)
        for idx in np.ndindex(pa.shape):
            up = [x.copy() for x in args]
            dn = [x.copy() for x in args]
            up[n][idx] += h
            dn[n][idx] -= h
            fd[idx] = (np.sum(dX * om.fwd(*up, incoming, bf16=False)) - np.sum(dX * om.fwd(*dn, incoming, bf16=False))) / (2 * h)
        err = np.max(np.abs(fd - grads[name])) / max(1e-12, np.max(np.abs(fd)))
        assert err < 1e-7, f"{name}: relative error {err}"


@pytest.mark.parametrize("incoming", [False, True])
def test_gradients_match_torch_autograd(incoming):
    pa, ga, pb, gb = _draw(2, 6, 3, seed=9)
    dX = np.random.default_rng(10).standard_normal(pa.shape)
    grads = om.bwd(pa, ga, pb, gb, dX, incoming, bf16=False)
    t = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (pa, ga, pb, gb)]
    a = torch.sigmoid(t[1]) * t[0]
    b = torch.sigmoid(t[3]) * t[2]
    X = torch.einsum("bkic,bkjc->bijc", a, b) if incoming else torch.einsum("bikc,bjkc->bijc", a, b)
    (X * torch.tensor(dX)).sum().backward()
    for name, tt in zip(("dPa", "dGa", "dPb", "dGb"), t):
        np.testing.assert_allclose(grads[name], tt.grad.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("incoming", [False, True])
def test_sampled_entries_equal_the_full_tensors(incoming):
    """The entry-wise evaluation used at sizes too large for the full oracle agrees with the full
    tensors at every entry of a small case (both directions, B = 2)."""
    pa, ga, pb, gb = _draw(2, 6, 3, seed=11)
    dX = np.random.default_rng(12).standard_normal(pa.shape)
    X = om.fwd(pa, ga, pb, gb, incoming)
    g = om.bwd(pa, ga, pb, gb, dX, incoming)
    idx = list(np.ndindex(pa.shape))
    s = om.sampled(pa, ga, pb, gb, dX, idx, incoming)
    np.testing.assert_allclose(s["X"], X.reshape(-1), rtol=1e-12, atol=1e-12)
    for k in ("dPa", "dGa", "dPb", "dGb"):
        np.testing.assert_allclose(s[k], g[k].reshape(-1), rtol=1e-12, atol=1e-12)
