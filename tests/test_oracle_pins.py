"""Pins of the FP64 oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to something external: central finite differences of
its own forward (gradients), PyTorch's scaled_dot_product_attention and its
float64 autograd (a library routine for ordinary attention with an additive
mask), closed forms (LSE = ln N, O = V[k*] for a single visible key, V = 1 =>
O = 1) and invariants of the mathematics (softmax rows sum to 1, dBias rows sum
to 0, dV columns sum to the dO columns, masked keys get no gradient).

Definition pinned (TurboPairFormer, arXiv 2610.05854v1, Abstract): per-slice
multi-head attention with a pair bias shared across slices, whose gradient is
the sum over slices of the per-slice score gradient.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _rand_case(B, S, N, H, d, seed, masked_keys=None, bias_std=1.0):
    rng = np.random.RandomState(seed)
    Q = rng.randn(B, S, N, H, d)
    K = rng.randn(B, S, N, H, d)
    V = rng.randn(B, S, N, H, d)
    dO = rng.randn(B, S, N, H, d)
    bias = bias_std * rng.randn(B, H, N, N)
    mask = None
    if masked_keys is not None:
        mask = np.zeros((B, S, N))
        for (b, i, k) in masked_keys:
            mask[b, i, k] = -np.inf
    return Q, K, V, bias, mask, dO


def _sdpa_reference(Q, K, V, bias, mask, scale, need_grad=False):
    """Ordinary attention per slice via torch SDPA (float64, CPU), bias+mask as attn_mask."""
    B, S, N, H, d = Q.shape
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=need_grad)
    q, k, v, bb = t(Q), t(K), t(V), t(bias)
    # [B,S,N,H,d] -> [B*S, H, N, d]
    perm = lambda x: x.permute(0, 1, 3, 2, 4).reshape(B * S, H, N, d)
    am = bb.unsqueeze(1).expand(B, S, H, N, N)
    if mask is not None:
        am = am + torch.tensor(mask, dtype=torch.float64)[:, :, None, None, :]
    am = am.reshape(B * S, H, N, N)
    o = torch.nn.functional.scaled_dot_product_attention(perm(q), perm(k), perm(v),
                                                         attn_mask=am, scale=scale)
    o = o.reshape(B, S, H, N, d).permute(0, 1, 3, 2, 4)
    return o, (q, k, v, bb)


def test_forward_matches_sdpa_with_bias_and_mask():
    Q, K, V, bias, mask, _ = _rand_case(2, 3, 7, 2, 4, seed=11, masked_keys=[(0, 1, 2), (1, 0, 6), (1, 2, 0)])
    scale = 1.0 / math.sqrt(4)
    O, LSE = oracle.fwd(Q, K, V, bias, mask, scale)
    ref, _ = _sdpa_reference(Q, K, V, bias, mask, scale)
    np.testing.assert_allclose(O, ref.detach().numpy(), rtol=1e-12, atol=1e-12)


def test_ordinary_attention_special_case():
    # one slice, no bias, no mask: plain softmax attention
    Q, K, V, _, _, _ = _rand_case(1, 1, 9, 3, 5, seed=3)
    bias = np.zeros((1, 3, 9, 9))
    O, _ = oracle.fwd(Q, K, V, bias, None)
    q = torch.tensor(Q[:, 0]).permute(0, 2, 1, 3)
    k = torch.tensor(K[:, 0]).permute(0, 2, 1, 3)
    v = torch.tensor(V[:, 0]).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v).permute(0, 2, 1, 3)
    np.testing.assert_allclose(O[:, 0], ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("B,S,N", [(2, 3, 9), (1, 37, 5)])  # S=37: several slices per dBias chunk
def test_gradients_match_torch_autograd(B, S, N):
    Q, K, V, bias, mask, dO = _rand_case(B, S, N, 2, 4, seed=5, masked_keys=[(0, 0, 3), (B - 1, 2, N - 1)])
    scale = 0.37  # a non-default scale also pins where scale enters
    g = oracle.bwd(Q, K, V, bias, mask, dO, scale)
    o, (q, k, v, bb) = _sdpa_reference(Q, K, V, bias, mask, scale, need_grad=True)
    (o * torch.tensor(dO)).sum().backward()
    np.testing.assert_allclose(g["dQ"], q.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dK"], k.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dV"], v.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dBias"], bb.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_gradients_central_finite_differences():
    B, S, N, H, d = 1, 2, 5, 2, 3
    Q, K, V, bias, mask, dO = _rand_case(B, S, N, H, d, seed=7, masked_keys=[(0, 1, 4)])
    scale = 1.0 / math.sqrt(d)
    g = oracle.bwd(Q, K, V, bias, mask, dO, scale)
    inputs = {"Q": Q, "K": K, "V": V, "bias": bias}
    grads = {"Q": g["dQ"], "K": g["dK"], "V": g["dV"], "bias": g["dBias"]}

    def loss(ins):
        O, _ = oracle.fwd(ins["Q"], ins["K"], ins["V"], ins["bias"], mask, scale)
        return float((O * dO).sum())

    h = 1e-5
    for name, x in inputs.items():
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            fd[idx] = (loss({**inputs, name: xp}) - loss({**inputs, name: xm})) / (2 * h)
        np.testing.assert_allclose(grads[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_softmax_rows_sum_to_one_and_masked_keys_get_zero():
    Q, K, V, bias, mask, dO = _rand_case(1, 2, 11, 2, 4, seed=9, masked_keys=[(0, 1, 3), (0, 1, 10)])
    for i in range(2):
        for h in range(2):
            P, _ = oracle.slice_matrices(Q, K, V, bias, mask, dO, 0, i, h)
            assert np.all(np.abs(P.sum(axis=1) - 1.0) < 1e-14)
            assert np.all(P >= 0.0)
    P, _ = oracle.slice_matrices(Q, K, V, bias, mask, dO, 0, 1, 1)
    assert np.all(P[:, 3] == 0.0) and np.all(P[:, 10] == 0.0)


def test_value_ones_gives_ones():
    Q, K, V, bias, mask, _ = _rand_case(1, 3, 8, 2, 5, seed=12, masked_keys=[(0, 2, 1)])
    O, _ = oracle.fwd(Q, K, np.ones_like(V), bias, mask)
    np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-14)


def test_lse_closed_forms():
    B, S, N, H, d = 1, 2, 6, 2, 3
    Z = np.zeros((B, S, N, H, d))
    _, LSE = oracle.fwd(Z, Z, Z, np.zeros((B, H, N, N)), np.zeros((B, S, N)))
    np.testing.assert_allclose(LSE, math.log(N), rtol=0, atol=1e-14)

    # a single visible key k*: LSE = S[j,k*] and O = V[k*]
    Q, K, V, bias, _, _ = _rand_case(B, S, N, H, d, seed=2)
    mask = np.full((B, S, N), -np.inf)
    kstar = 4
    mask[:, :, kstar] = 0.0
    O, LSE = oracle.fwd(Q, K, V, bias, mask, 0.5)
    for i in range(S):
        for h in range(H):
            for j in range(N):
                s = 0.5 * Q[0, i, j, h] @ K[0, i, kstar, h] + bias[0, h, j, kstar]
                assert abs(LSE[0, i, h, j] - s) < 1e-12
                np.testing.assert_allclose(O[0, i, j, h], V[0, i, kstar, h], rtol=0, atol=1e-14)


def test_bias_row_shift_invariance():
    Q, K, V, bias, mask, _ = _rand_case(1, 3, 7, 2, 4, seed=4, masked_keys=[(0, 0, 2)])
    O1, L1 = oracle.fwd(Q, K, V, bias, mask)
    shift = np.random.RandomState(0).randn(1, 2, 7, 1)  # per (h, j) constant over keys
    O2, L2 = oracle.fwd(Q, K, V, bias + shift, mask)
    np.testing.assert_allclose(O2, O1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2 - L1, np.broadcast_to(shift[:, None, :, :, 0], L1.shape), atol=1e-12)


def test_dbias_is_slice_sum_of_dS_and_rows_sum_to_zero():
    B, S, N, H, d = 2, 4, 6, 2, 3
    Q, K, V, bias, mask, dO = _rand_case(B, S, N, H, d, seed=8, masked_keys=[(1, 3, 5)])
    g = oracle.bwd(Q, K, V, bias, mask, dO)
    for b in range(B):
        for h in range(H):
            acc = np.zeros((N, N))
            for i in range(S):
                _, dS = oracle.slice_matrices(Q, K, V, bias, mask, dO, b, i, h)
                np.testing.assert_allclose(dS.sum(axis=1), 0.0, atol=1e-13)
                acc += dS
            np.testing.assert_allclose(g["dBias"][b, h], acc, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dBias"].sum(axis=-1), 0.0, atol=1e-12)


def test_dv_column_sums_and_masked_key_gradients():
    B, S, N, H, d = 1, 3, 8, 2, 4
    masked = [(0, 0, 1), (0, 1, 1), (0, 2, 1), (0, 2, 6)]  # key 1 masked in every slice
    Q, K, V, bias, mask, dO = _rand_case(B, S, N, H, d, seed=10, masked_keys=masked)
    g = oracle.bwd(Q, K, V, bias, mask, dO)
    np.testing.assert_allclose(g["dV"].sum(axis=2), dO.sum(axis=2), rtol=1e-12, atol=1e-12)
    for (b, i, k) in masked:
        assert np.all(g["dK"][b, i, k] == 0.0) and np.all(g["dV"][b, i, k] == 0.0)
    assert np.all(g["dBias"][:, :, :, 1] == 0.0)


def test_fully_masked_slice_contributes_nothing():
    B, S, N, H, d = 1, 3, 5, 2, 3
    Q, K, V, bias, _, dO = _rand_case(B, S, N, H, d, seed=13)
    mask = np.zeros((B, S, N))
    mask[:, 1, :] = -np.inf
    O, LSE = oracle.fwd(Q, K, V, bias, mask)
    assert np.all(O[:, 1] == 0.0) and np.all(np.isneginf(LSE[:, 1]))
    g = oracle.bwd(Q, K, V, bias, mask, dO)
    for name in ("dQ", "dK", "dV"):
        assert np.all(g[name][:, 1] == 0.0)
    keep = [0, 2]
    g2 = oracle.bwd(Q[:, keep], K[:, keep], V[:, keep], bias, mask[:, keep], dO[:, keep])
    np.testing.assert_allclose(g["dBias"], g2["dBias"], rtol=1e-13, atol=1e-14)


def test_exact_D_and_thread_count_independence():
    Q, K, V, bias, mask, dO = _rand_case(1, 5, 7, 2, 3, seed=14, masked_keys=[(0, 4, 0)])
    g1 = oracle.bwd(Q, K, V, bias, mask, dO, nthreads=1)
    g4 = oracle.bwd(Q, K, V, bias, mask, dO, nthreads=4)
    for k in g1:
        assert np.array_equal(g1[k], g4[k]), k
    # D is the row sum of dO * O with the exact forward output
    O, _ = oracle.fwd(Q, K, V, bias, mask)
    np.testing.assert_allclose(g1["D"], np.einsum("bsnhc,bsnhc->bshn", dO, O), rtol=1e-12, atol=1e-13)


def test_golden_regression_fixture():
    import json, os
    from tests.golden.make_golden import compute
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny.json")
    want = json.load(open(path))["values"]
    got = compute()
    for k in want:
        np.testing.assert_allclose(np.array(got[k]), np.array(want[k]), rtol=1e-14, atol=1e-15, err_msg=k)


def test_dbias_rows_agree_with_torch_autograd():
    # the row-wise dBias routine (used at sizes where the full backward is too slow)
    Q, K, V, bias, mask, dO = _rand_case(2, 6, 7, 2, 3, seed=21, masked_keys=[(0, 2, 6), (1, 5, 0)])
    o, (q, k, v, bb) = _sdpa_reference(Q, K, V, bias, mask, 1.0 / math.sqrt(3), need_grad=True)
    (o * torch.tensor(dO)).sum().backward()
    rows = [(0, 0, 0), (0, 1, 6), (1, 1, 3), (1, 0, 5)]
    got = oracle.dbias_rows(Q, K, V, bias, mask, dO, rows)
    for r, (b, h, j) in enumerate(rows):
        np.testing.assert_allclose(got[r], bb.grad.numpy()[b, h, j], rtol=1e-10, atol=1e-12)
