"""GPU parity of the triangle multiplicative update against the FP64 oracle (oracle/trimul.py).

The CUDA path runs through the C ABI (tri_mul_fwd / tri_mul_bwd via the ctypes binding); the oracle
gets the same seeded BF16 inputs. Small shapes compare every element of every output; the crop-768
workload compares whole channels (each channel of the update is an independent matrix product, so a
channel slice of the inputs gives the oracle's exact value for that channel).

Tolerances, derived from the arithmetic and computed from oracle values only:
- gated operands A, Bm: the kernel evaluates sigmoid(G) P in FP32 with a relative error below
  GATE_REL = 2^-17 (|G| < 16: the exponential's error grows with |G|), then rounds to BF16. Its BF16
  value therefore equals the FP64 one except where the exact value lies within GATE_REL of a
  rounding midpoint ("ambiguous" elements, about 0.3 %), where it may be one ulp away. Checked
  exactly: equal everywhere else, at most one ulp at ambiguous elements.
- X = sum_k a b with FP32 accumulation of exact BF16 products: per element
      |X - ref| <= ulp_bf16(ref) + GAMMA * sum_k |a||b| + sum_k (amb_a ulp(a) |b| + |a| amb_b ulp(b))
  (output rounding; accumulation, GAMMA = N 2^-22, four times the textbook bound since the
  tensor cores' addition order is not specified; one ulp for every ambiguous operand);
- dA = dX Bm likewise (dX is exact BF16), dB = dX^T A, then dP = dA sigmoid(G) and
  dG = dA P sigmoid(G)(1 - sigmoid(G)) in FP32: the dA bound carried through the factors, the
  FP32 sigmoid's relative error SIG_REL = 2^-19 (fast exponential and reciprocal: a few ulp plus
  about one ulp per unit of |G|, for the |G| < 6 of these inputs; and its effect on 1 - sigmoid,
  relative SIG_REL sigmoid / (1 - sigmoid)), a few FP32 roundings, and the output ulp.
Whole-tensor relative RMSE <= 2e-3 is checked as well.
"""
import numpy as np
import pytest
import torch

from bwd_tri_attn_gb300 import workloads as wl
from oracle import trimul as om
from tests.parity_util import rmse_rel, ulp_bf16

pytestmark = pytest.mark.gpu

RMSE_TOL = 2e-3
GATE_REL = 2.0 ** -17
SIG_REL = 2.0 ** -19


def sig_rel(g):
    """Relative error bound of the kernels' FP32 sigmoid: the fast exponential's documented
    2 + 1.173 |x| ulp, the fast reciprocal's 2 ulp and the add, with a factor 2 of margin."""
    return 2.0 * (5.0 + 1.2 * np.abs(g)) * 2.0 ** -24


def _lib():
    from bwd_tri_attn_gb300 import _build, binding
    _build.build()
    binding.load()
    return binding


def _f64(t):
    return t.detach().to("cpu").double().numpy()


PAIR, CM = 0, 1  # layouts of the projections and their gradients
PROJ = ("Pa", "Ga", "Pb", "Gb")
GRADS = ("dPa", "dGa", "dPb", "dGb")


def run_cuda(x, incoming, layout=PAIR):
    """One forward + backward through the C ABI. ``x`` holds pair-layout projections; with the
    channel-major layout they are handed over as [B, C, N, N] and the gradients mapped back."""
    tb = _lib()
    d = {k: v.cuda() for k, v in x.items()}
    if layout == CM:
        d = {k: (v.permute(0, 3, 1, 2) if k in PROJ else v) for k, v in d.items()}
    d = {k: v.contiguous() for k, v in d.items()}
    X, A, Bm = tb.mul_forward(d["Pa"], d["Ga"], d["Pb"], d["Gb"], incoming=incoming, layout=layout)
    dPa, dGa, dPb, dGb = tb.mul_backward(d["Pa"], d["Ga"], d["Pb"], d["Gb"], A, Bm, d["dX"], incoming=incoming,
                                         layout=layout)
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
    out = dict(X=X, A=A, Bm=Bm, dPa=dPa, dGa=dGa, dPb=dPb, dGb=dGb)
    if layout == CM:
        out = {k: (v.permute(0, 2, 3, 1) if k in GRADS else v) for k, v in out.items()}
    return {k: v.contiguous().cpu() for k, v in out.items()}


def channel_major(a):
    """[B, N, N, C] -> [B, C, N, N]."""
    return np.ascontiguousarray(np.moveaxis(a, -1, 1))


def ambiguous(exact, rel=GATE_REL):
    """Elements whose exact value lies within `rel` (relative) of a BF16 rounding midpoint."""
    a = np.abs(exact)
    u = ulp_bf16(exact)
    frac = np.mod(a, u) / u  # position inside the BF16 interval, in ulps
    return (np.abs(frac - 0.5) * u <= rel * a) & (a > 0)


def oracle_all(x, incoming, layout=PAIR):
    """Oracle outputs (channel-major X, A, Bm; pair-layout gradients) and a per-element tolerance
    for each, from the oracle's values only. The saved operands A, Bm hold the pair axes swapped
    for the incoming update in the pair layout only."""
    pa, ga, pb, gb = (_f64(x[k]) for k in ("Pa", "Ga", "Pb", "Gb"))
    dX = np.moveaxis(_f64(x["dX"]), 1, -1)  # channel-major -> pair layout
    a, b = om.gated(pa, ga), om.gated(pb, gb)
    # FP32 gating error: the sigmoid's (grows with |G|) and the product's rounding
    amb_a = ambiguous(om.gated(pa, ga, bf16=False), np.maximum(GATE_REL, 4 * sig_rel(ga)))
    amb_b = ambiguous(om.gated(pb, gb, bf16=False), np.maximum(GATE_REL, 4 * sig_rel(gb)))
    da_ulp, db_ulp = amb_a * ulp_bf16(a), amb_b * ulp_bf16(b)
    N = pa.shape[1]
    gamma = N * 2.0 ** -22
    # bounds go through BLAS-backed contractions (they are tolerances, not the oracle's arithmetic)
    spec = "bkic,bkjc->bijc" if incoming else "bikc,bjkc->bijc"
    c = lambda u, v: np.einsum(spec, u, v, optimize=True)
    X = om.fwd(pa, ga, pb, gb, incoming)
    tX = ulp_bf16(X) + gamma * c(np.abs(a), np.abs(b)) + c(da_ulp, np.abs(b)) + c(np.abs(a), db_ulp)
    g = om.bwd(pa, ga, pb, gb, dX, incoming)
    # bounds on dA = dX Bm and dB = dX^T A (the same contractions as the oracle's gradients)
    if incoming:
        tdA = np.einsum("bijc,bkjc->bkic", np.abs(dX), gamma * np.abs(b) + db_ulp, optimize=True)
        tdB = np.einsum("bijc,bkic->bkjc", np.abs(dX), gamma * np.abs(a) + da_ulp, optimize=True)
    else:
        tdA = np.einsum("bijc,bjkc->bikc", np.abs(dX), gamma * np.abs(b) + db_ulp, optimize=True)
        tdB = np.einsum("bijc,bikc->bjkc", np.abs(dX), gamma * np.abs(a) + da_ulp, optimize=True)
    sa, sb = om.sigmoid(ga), om.sigmoid(gb)
    tol = {"X": tX}
    for name, t, s_, p, g_ in (("a", tdA, sa, pa, ga), ("b", tdB, sb, pb, gb)):
        dP, dG = g["dP" + name], g["dG" + name]
        r = np.maximum(SIG_REL, sig_rel(g_))
        with np.errstate(divide="ignore"):
            amp = s_ / (1 - s_)  # relative error growth of 1 - sigmoid (infinite where it is 0 in FP64)
        tol["dP" + name] = ulp_bf16(dP) + t * s_ + (r + 2.0 ** -23) * np.abs(dP)
        # (where 1 - sigmoid is 0 in FP64, dG is 0 and so is the kernel's: no relative term)
        with np.errstate(invalid="ignore"):
            rel_g = np.where(np.abs(dG) > 0, (r * (1 + amp) + 2.0 ** -22) * np.abs(dG), 0.0)
        tol["dG" + name] = ulp_bf16(dG) + t * np.abs(p) * s_ * (1 - s_) + rel_g
    if incoming and layout == PAIR:  # the stored operands hold the pair axes swapped
        a, b = np.swapaxes(a, 1, 2), np.swapaxes(b, 1, 2)
        amb_a, amb_b = np.swapaxes(amb_a, 1, 2), np.swapaxes(amb_b, 1, 2)
    out = dict(X=channel_major(X), A=channel_major(a), Bm=channel_major(b), **g)
    tol["X"] = channel_major(tol["X"])
    amb = dict(A=channel_major(amb_a), Bm=channel_major(amb_b))
    return out, tol, amb


def check_operand(got, want, amb, what):
    got, want = _f64(got), np.asarray(want)
    diff = np.abs(got - want)
    assert np.all(diff[~amb] == 0), f"{what}: {np.count_nonzero(diff[~amb])} unambiguous elements differ"
    assert np.all(diff[amb] <= ulp_bf16(want[amb])), f"{what}: an ambiguous element is more than one ulp off"


def check_value(got, want, tol, what):
    got, want = _f64(got), np.asarray(want, dtype=np.float64)
    r = rmse_rel(got, want)
    assert r <= RMSE_TOL, f"{what}: relative RMSE {r:.3e}"
    ratio = np.abs(got - want) / tol
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert ratio[worst] <= 1.0, (f"{what}: |err| {abs(got[worst] - want[worst]):.3g} exceeds its bound "
                                 f"{tol[worst]:.3g} at {worst}")
    return float(ratio.max())


def check_all(got, ref, tol, amb):
    check_operand(got["A"], ref["A"], amb["A"], "A")
    check_operand(got["Bm"], ref["Bm"], amb["Bm"], "Bm")
    for k in ("X", "dPa", "dGa", "dPb", "dGb"):
        check_value(got[k], ref[k], tol[k], k)


SMALL = [(1, 16, 8, 10), (2, 72, 24, 11), (1, 136, 72, 14), (1, 264, 16, 15)]


@pytest.mark.parametrize("layout", [PAIR, CM])
@pytest.mark.parametrize("incoming", [False, True])
@pytest.mark.parametrize("B,N,C,seed", SMALL)
def test_full_parity_small(B, N, C, seed, incoming, layout):
    x = wl.make_mul_inputs(B, N, C, seed)
    got = run_cuda(x, incoming, layout)
    check_all(got, *oracle_all(x, incoming, layout))


@pytest.mark.parametrize("layout", [PAIR, CM])
@pytest.mark.parametrize("incoming", [False, True])
def test_crop768_sampled_channels(incoming, layout):
    """The full crop-768 workload (B=1, N=768, C=128) in one launch configuration; three channels
    (in both gating channel groups and in three of the gradient kernel's groups) checked whole."""
    w = wl.MUL_CROP768
    x = wl.mul_inputs_for(w)
    got = run_cuda(x, incoming, layout)
    cs = [0, 77, 127]
    sl = {k: (v[..., cs] if k != "dX" else v[:, cs]) for k, v in x.items()}
    sub = {k: (v[:, cs] if k in ("X", "A", "Bm") else v[..., cs]) for k, v in got.items()}
    check_all(sub, *oracle_all(sl, incoming, layout))


def test_zero_projection_gives_exact_zeros():
    """P_a = 0: a = 0, so X = 0 and dG_a, dP_b, dG_b vanish exactly (dB = dX^T A = 0); dP_a =
    dA sigmoid(G_a) still carries values (checked against the oracle)."""
    x = wl.make_mul_inputs(1, 96, 16, 16)
    x["Pa"] = torch.zeros_like(x["Pa"])
    got = run_cuda(x, False, CM)
    assert torch.count_nonzero(got["A"]) == 0 and torch.count_nonzero(got["X"]) == 0
    assert torch.count_nonzero(got["dGa"]) == 0 and torch.count_nonzero(got["dPb"]) == 0
    assert torch.count_nonzero(got["dGb"]) == 0  # dG_b = dB P_b s(1-s), dB = dX^T A = 0
    ref, tol, _ = oracle_all(x, False)
    check_value(got["dPa"], ref["dPa"], tol["dPa"], "dPa")


@pytest.mark.parametrize("layout", [PAIR, CM])
@pytest.mark.parametrize("incoming", [False, True])
def test_deterministic(incoming, layout):
    x = wl.make_mul_inputs(1, 200, 32, 17)
    a, b = run_cuda(x, incoming, layout), run_cuda(x, incoming, layout)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_layouts_agree_bitwise_outgoing():
    """Outgoing update: the channel-major path (gating gradient in the contraction's epilogue) and
    the pair path (FP32 dA, dB, then the layout-changing gradient kernel) run the same products in
    the same order and the same element-wise arithmetic: identical bits."""
    x = wl.make_mul_inputs(1, 136, 24, 20)
    a, b = run_cuda(x, False, PAIR), run_cuda(x, False, CM)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_incoming_is_outgoing_of_transposed_inputs():
    """The incoming update on P equals the outgoing update on the pair-transposed P (both computed on
    the GPU; exact, since both run the same sums in the same order)."""
    x = wl.make_mul_inputs(1, 80, 16, 18)
    t = {k: (v.transpose(1, 2).contiguous() if k != "dX" else v) for k, v in x.items()}
    a, b = run_cuda(x, True), run_cuda(t, False)
    assert torch.equal(a["X"], b["X"]) and torch.equal(a["A"], b["A"])
    for k in ("dPa", "dGa", "dPb", "dGb"):
        assert torch.equal(a[k], b[k].transpose(1, 2)), k


def test_device_errors_before_launch():
    tb = _lib()
    from bwd_tri_attn_gb300.binding import MulShape, TriAttnError
    x = {k: v.cuda() for k, v in wl.make_mul_inputs(1, 64, 8, 19).items()}
    X, A, Bm = tb.mul_forward(x["Pa"], x["Ga"], x["Pb"], x["Gb"])
    shape = MulShape(1, 64, 8, 0)
    need = tb.tri_mul_bwd_workspace_size(shape)
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    outs = [torch.empty_like(x["Pa"]) for _ in range(4)]
    with pytest.raises(TriAttnError) as e:
        tb.tri_mul_bwd(shape, x["Pa"], x["Ga"], x["Pb"], x["Gb"], A, Bm, x["dX"], *outs, small)
    assert e.value.code == -3
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0


# ---------------------------------------------------------------- edge cases: sizes and gate range
@pytest.mark.parametrize("layout", [PAIR, CM])
@pytest.mark.parametrize("incoming", [False, True])
def test_max_channels_full_oracle(incoming, layout):
    """C = TRI_MUL_MAX_C = 1024 (16 gating channel groups, 32 gradient groups) on a small N."""
    x = wl.make_mul_inputs(1, 24, 1024, 21)
    got = run_cuda(x, incoming, layout)
    check_all(got, *oracle_all(x, incoming, layout))


def test_largest_batch_times_channels():
    """B * C at its limit region (B = 64, C = 1016: 65,024 matrix products in one launch)."""
    x = wl.make_mul_inputs(64, 16, 1016, 22)
    for layout in (PAIR, CM):
        got = run_cuda(x, False, layout)
        check_all(got, *oracle_all(x, False, layout))


@pytest.mark.parametrize("incoming", [False, True])
def test_max_n_sampled_entries(incoming):
    """N = TRI_MUL_MAX_N = 4096 (16 x 32 output tiles per channel, 64 K steps): 48 entries of X and
    of every gradient against the oracle's entry-wise evaluation, with the per-entry bound of the
    full-oracle tests (output ulp, FP32 accumulation over N terms, ambiguous operand roundings,
    the sigmoid's error)."""
    B, N, C = 1, 4096, 8
    x = wl.make_mul_inputs(B, N, C, 23)
    got = run_cuda(x, incoming, CM)
    g = np.random.default_rng(24)
    idx = [(0, 0, 0, 0), (0, N - 1, N - 1, C - 1), (0, 0, N - 1, 3), (0, N - 1, 0, 4)]
    idx += [(0, int(a), int(b_), int(c)) for a, b_, c in zip(g.integers(0, N, 44), g.integers(0, N, 44),
                                                               g.integers(0, C, 44))]
    f = {k: _f64(v) for k, v in x.items()}
    dX = np.moveaxis(f["dX"], 1, -1)
    ref = om.sampled(f["Pa"], f["Ga"], f["Pb"], f["Gb"], dX, idx, incoming)
    gamma = N * 2.0 ** -22
    for n, (b, i, j, c) in enumerate(idx):
        # the rows and columns the entry touches, gated exactly and in BF16
        def rows(P, G, axis_first, k):
            sl = (b, slice(None), k, c) if axis_first else (b, k, slice(None), c)
            return om.gated(P[sl], G[sl]), ambiguous(om.gated(P[sl], G[sl], bf16=False))
        a_r, amb_a = rows(f["Pa"], f["Ga"], incoming, i)
        b_r, amb_b = rows(f["Pb"], f["Gb"], incoming, j)
        tol = (ulp_bf16(ref["X"][n]) + gamma * np.dot(np.abs(a_r), np.abs(b_r))
               + np.dot(amb_a * ulp_bf16(a_r), np.abs(b_r)) + np.dot(np.abs(a_r), amb_b * ulp_bf16(b_r)))
        err = abs(float(got["X"][b, c, i, j]) - ref["X"][n])
        assert err <= tol, f"X{(b, i, j, c)}: |err| {err:.3g} > {tol:.3g}"
        # gradients at projection entry [b, i, j, c]: bound on dA / dB from the terms they sum
        if incoming:
            ta, tb = rows(f["Pb"], f["Gb"], False, i), rows(f["Pa"], f["Ga"], False, i)
            dxa, dxb = np.abs(dX[b, j, :, c]), np.abs(dX[b, :, j, c])
        else:
            ta, tb = rows(f["Pb"], f["Gb"], True, j), rows(f["Pa"], f["Ga"], True, j)
            dxa, dxb = np.abs(dX[b, i, :, c]), np.abs(dX[b, :, i, c])
        tda = np.dot(dxa, gamma * np.abs(ta[0]) + ta[1] * ulp_bf16(ta[0]))
        tdb = np.dot(dxb, gamma * np.abs(tb[0]) + tb[1] * ulp_bf16(tb[0]))
        for name, td, P, G in (("a", tda, f["Pa"], f["Ga"]), ("b", tdb, f["Pb"], f["Gb"])):
            s_ = om.sigmoid(G[b, i, j, c])
            r = sig_rel(G[b, i, j, c])
            dP, dG = ref["dP" + name][n], ref["dG" + name][n]
            tolP = ulp_bf16(dP) + td * s_ + (r + 2.0 ** -23) * abs(dP)
            tolG = ulp_bf16(dG) + td * abs(P[b, i, j, c]) * s_ * (1 - s_) + (r * (1 + s_ / (1 - s_)) + 2.0 ** -22) * abs(dG)
            for k, want, t in (("dP" + name, dP, tolP), ("dG" + name, dG, tolG)):
                e = abs(float(got[k][b, i, j, c]) - want)
                assert e <= t, f"{k}{(b, i, j, c)}: |err| {e:.3g} > {t:.3g}"


@pytest.mark.parametrize("layout", [PAIR, CM])
def test_saturated_gates(layout):
    """Gate logits N(0, 12) (|G| up to about 55: sigmoid saturates to 0 and 1 in FP32): the gated
    operands still match the FP64 rounding away from ambiguous entries, and X and the gradients
    stay within their bounds, where 1 - sigmoid loses its relative precision."""
    x = wl.make_mul_inputs(1, 72, 16, 25, gate_std=12.0)
    assert float(x["Ga"].float().abs().max()) < 80.0  # inside the kernels' documented gate range
    got = run_cuda(x, False, layout)
    check_all(got, *oracle_all(x, False, layout))
