"""GPU parity: the CUDA path against the FP64 oracle, element by element.

Gate: relative RMSE <= 2e-3 for O, dQ, dK, dV and dBias; LSE to
FP32 accuracy; residual compensation lowers dQ, dK and dBias error; all
outputs bitwise identical across repeated calls. Beside the RMSE, every
compared element must lie within one BF16 ulp of the oracle plus a small
fraction of the tensor's rms (tests/parity_util.py), which a single wrong store
fails.

Small and ragged shapes are compared on every element against the full
oracle; the crop-size shapes run at full size on the GPU and are compared on
sampled slices (O, LSE, dQ, dK, dV) and sampled bias rows (dBias), which the
oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from bwd_tri_attn_gb300 import workloads as wl
from tests.parity_util import (RMSE_REL_TOL, boundary_slices, check_elementwise, check_lse, f64, oracle_full,
                               rmse_rel, run_cuda)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bwd_tri_attn_gb300 import _build, binding
    _build.build()
    binding.load()


def _compare_all(got, want, what, tol=RMSE_REL_TOL):
    errs = {}
    for k in ("O", "dQ", "dK", "dV", "dBias"):
        errs[k] = rmse_rel(f64(got[k]), want[k])
    check_lse(f64(got["LSE"]), want["LSE"], what)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{what}: RMSE above {tol}: {errs}"
    for k in ("O", "dQ", "dK", "dV", "dBias"):
        check_elementwise(f64(got[k]), want[k], f"{what} {k}")
    return errs


SMALL = [
    ("tiny", dict(B=1, S=32, N=32, H=2, d=16, seed=0, mask=("none",))),
    ("pad128", dict(B=1, S=128, N=128, H=4, d=32, seed=1, value_std=0.5, mask=("tail", 13))),
    ("ragged200_d32", dict(B=2, S=3, N=200, H=3, d=32, seed=5, mask=("random", 0.1))),
    ("ragged77_d16", dict(B=1, S=5, N=77, H=2, d=16, seed=6, mask=("tail", 7))),
    ("tile_plus_one", dict(B=1, S=3, N=129, H=1, d=32, seed=7, mask=("zeros",))),
    ("two_tiles_d16", dict(B=1, S=9, N=256, H=2, d=16, seed=8, mask=("random", 0.05))),
    ("single_key", dict(B=1, S=4, N=1, H=2, d=32, seed=9, mask=("none",))),
    ("batch3", dict(B=3, S=6, N=48, H=1, d=16, seed=10, mask=("random", 0.2))),
]


@pytest.mark.parametrize("name,cfg", SMALL, ids=[s[0] for s in SMALL])
def test_parity_full_oracle(name, cfg):
    x = wl.make_inputs(**cfg)
    got = run_cuda(x)
    want = oracle_full(x)
    if cfg["N"] == 1:
        # one key: P = 1, so O = V and dV = dO exactly; dQ = dK = dBias = 0 up to the
        # rounding difference between two FP32 evaluations of dO.V
        assert torch.equal(got["O"], x["V"]) and torch.equal(got["dV"], x["dO"])
        for k in ("dQ", "dK", "dBias"):
            assert got[k].float().abs().max().item() <= 1e-4
        return
    _compare_all(got, want, name)
    # Ores carries the output-rounding residual: O + Ores is closer to the exact output
    e_plain = rmse_rel(f64(got["O"]), want["O"])
    e_comp = rmse_rel(f64(got["O"]) + f64(got["Ores"]), want["O"])
    assert e_comp < 0.2 * e_plain


def test_fully_masked_slice():
    x = wl.make_inputs(B=1, S=4, N=40, H=2, d=32, seed=11, mask=("slices", [1]))
    got = run_cuda(x)
    want = oracle_full(x)
    assert torch.count_nonzero(got["O"][:, 1]) == 0
    assert torch.all(torch.isneginf(got["LSE"][:, 1]))
    for k in ("dQ", "dK", "dV"):
        assert torch.count_nonzero(got[k][:, 1]) == 0
    _compare_all(got, want, "fully_masked_slice")


@pytest.mark.parametrize("d", [16, 32])
def test_lazy_max_raised_in_later_key_tiles(d):
    # a bias ramp over the keys lifts every key tile's row max by 6.4 over the previous one,
    # more than the forward's lazy-max threshold (8 ln 2 = 5.5): each row's reference max is
    # raised, and O rescaled in TMEM, at every key tile after the first
    x = wl.make_inputs(B=1, S=6, N=512, H=2, d=d, seed=21, mask=("random", 0.05))
    ramp = 0.05 * torch.arange(512, dtype=torch.float32)
    x["bias"] = (x["bias"].float() + ramp).to(torch.bfloat16)
    got = run_cuda(x)
    want = oracle_full(x)
    _compare_all(got, want, f"bias_ramp_d{d}")


@pytest.mark.parametrize("d", [16, 32])
def test_rows_without_visible_keys_in_first_key_tiles(d):
    # slices whose first one or two key tiles are fully masked: the forward takes the row's
    # reference max only from the first key tile that has a visible key
    x = wl.make_inputs(B=1, S=5, N=300, H=2, d=d, seed=22, mask=("zeros",))
    m = x["mask"].float()
    m[:, 0, :128] = float("-inf")
    m[:, 2, :128] = float("-inf")
    m[:, 3, :256] = float("-inf")
    x["mask"] = m.to(torch.bfloat16)
    got = run_cuda(x)
    want = oracle_full(x)
    _compare_all(got, want, f"masked_first_tiles_d{d}")


def test_ragged_slice_groups_across_units():
    # more work units than SMs (4 x 2 x 4 x 6 = 192), with S = 7 not a multiple of the forward's
    # slice group: a CTA walks units with four and with three slices in turn, so its per-slice Q
    # buffers and per-warpgroup O barriers change how many slices they serve between units
    x = wl.make_inputs(B=4, S=7, N=768, H=4, d=32, seed=23, mask=("tail", 20))
    got = run_cuda(x)
    want = oracle_full(x)
    _compare_all(got, want, "ragged_units")


MAXN = [
    ("n1024_d32", dict(B=1, S=3, N=1024, H=2, d=32, seed=41, mask=("tail", 30))),
    ("n1000_d16", dict(B=1, S=2, N=1000, H=3, d=16, seed=42, mask=("random", 0.05))),
]


@pytest.mark.parametrize("name,cfg", MAXN, ids=[m[0] for m in MAXN])
def test_largest_key_count_full_oracle(name, cfg):
    # N up to the supported maximum of 1024: eight key tiles, so the backward runs its largest
    # cluster (eight CTAs, each owning 16 dQ rows of a step); N = 1000 leaves a ragged last tile
    x = wl.make_inputs(**cfg)
    got = run_cuda(x)
    want = oracle_full(x)
    _compare_all(got, want, name)
    end = run_cuda(x, node=1)
    for k in ("O", "LSE", "Ores", "dQ", "dK", "dV", "dBias"):
        assert torch.equal(end[k].view(torch.uint8), got[k].view(torch.uint8)), f"{name}: {k} differs by layout"


@pytest.mark.parametrize("d", [16, 32])
def test_largest_head_count_full_oracle(d):
    # H = 256, the supported maximum: 16 KB (d = 32) between a row's heads in the pair tensors,
    # and the D kernel's per-block head buffer at its largest
    x = wl.make_inputs(B=1, S=2, N=130, H=256, d=d, seed=43 + d, mask=("random", 0.1))
    got = run_cuda(x)
    want = oracle_full(x)
    _compare_all(got, want, f"h256_d{d}")


def test_pair_tensors_above_2_31_elements():
    # B*S*N*H*d = 257 * 1024 * 256 * 32 > 2^31 elements per pair tensor (4.3 GB in BF16, about
    # 45 GB on the device in all): element offsets need 64 bits everywhere. The inputs are drawn on
    # the device. A head's O, LSE, dQ, dK and dV depend only on that head's inputs and bias, so
    # sampled (slice, head) pairs are checked against the oracle on that sub-problem; dBias rows,
    # which sum over all slices, are checked for two heads over all 257 slices.
    import oracle
    from bwd_tri_attn_gb300 import binding as tb

    B, S, N, H, d = 1, 257, 1024, 256, 32
    assert B * S * N * H * d > 2 ** 31
    gen = torch.Generator(device="cuda").manual_seed(61)

    def normal(shape):
        return torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)

    x = {k: normal((B, S, N, H, d)) for k in ("Q", "K", "V", "dO")}
    x["bias"] = normal((B, H, N, N))
    x["mask"] = wl.make_mask(("tail", 30), B, S, N, torch.Generator().manual_seed(61)).cuda()
    O, LSE, Ores = tb.forward(x["Q"], x["K"], x["V"], x["bias"], x["mask"])
    dQ, dK, dV, dBias = tb.backward(x["Q"], x["K"], x["V"], x["bias"], x["mask"], O, Ores, LSE, x["dO"])
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0

    sl, heads = [0, 129, 256], [0, 255]

    def sub(t):  # [B, S, N, H, d] -> sampled slices and heads, on the host
        return t[:, sl][:, :, :, heads].cpu()

    xs = {k: sub(x[k]) for k in ("Q", "K", "V", "dO")}
    xs["bias"] = x["bias"][:, heads].cpu()
    xs["mask"] = x["mask"][:, sl].cpu()
    want = oracle_full(xs)
    for k, t in (("O", O), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        e = rmse_rel(f64(sub(t)), want[k])
        assert e <= RMSE_REL_TOL, f"{k} RMSE {e}"
    check_lse(f64(LSE[:, sl][:, :, heads].cpu()), want["LSE"], "above_2_31")

    xh = {k: x[k][:, :, :, heads].cpu() for k in ("Q", "K", "V", "dO")}
    rows = [(0, 0, 5), (0, 1, 517), (0, 1, N - 1)]
    want_rows = oracle.dbias_rows(xh["Q"], xh["K"], xh["V"], xs["bias"], x["mask"].cpu(), xh["dO"], rows)
    got_rows = np.stack([f64(dBias[b, heads[h], j].cpu()) for (b, h, j) in rows])
    e = rmse_rel(got_rows, want_rows)
    assert e <= RMSE_REL_TOL, f"dBias sampled-row RMSE {e}"
    del x, O, LSE, Ores, dQ, dK, dV, dBias
    torch.cuda.empty_cache()


def test_scale_argument_is_used():
    x = wl.make_inputs(B=1, S=4, N=64, H=2, d=16, seed=12, mask=("tail", 3))
    got = run_cuda(x, scale=0.37)
    want = oracle_full(x, scale=0.37)
    _compare_all(got, want, "scale")


# The FP16 operand staging against the whole BF16 range: the same problem with one tensor
# scaled by a power of two (gradients of a loss scaled far down or up, tiny values, large
# activations). Relative errors must not move.
RANGE = [
    ("dO_2^-20", {"dO": -20}),
    ("dO_2^-12", {"dO": -12}),
    ("dO_2^8", {"dO": 8}),
    ("V_2^-16", {"V": -16}),
    ("V_2^16", {"V": 16}),
    ("dO_2^14", {"dO": 14}),
    ("Q_2^-16_K_2^10", {"Q": -16, "K": 10}),
    ("all_2^-30", {"Q": -30, "K": -30, "V": -30, "dO": -30}),
]


@pytest.mark.parametrize("d", [16, 32])
@pytest.mark.parametrize("name,exps", RANGE, ids=[r[0] for r in RANGE])
def test_input_range_full_oracle(name, exps, d):
    # ragged: N = 200 (two key tiles, the second partial), S = 7, random key mask
    x = wl.scale_pow2(wl.make_inputs(B=1, S=7, N=200, H=2, d=d, seed=51, mask=("random", 0.1)), exps)
    got = run_cuda(x)
    want = oracle_full(x)
    _compare_all(got, want, f"{name}_d{d}")


@pytest.mark.parametrize("name,exps", RANGE[:4], ids=[r[0] for r in RANGE[:4]])
def test_input_range_crop384_sampled(name, exps):
    w = wl.CROP384
    x = wl.scale_pow2(wl.inputs_for(w), exps)
    N = w.N
    rows = [(0, h, j) for h in range(w.H) for j in (1, N - 2)]
    _sampled_check(x, _split_slices(w)[:12], rows, f"crop384_{name}")


ABLATION = [wl.CROP384, wl.CROP640_D16, wl.CROP640_D32, wl.CROP768]


@pytest.mark.parametrize("w", ABLATION, ids=[w.name for w in ABLATION])
def test_residual_compensation_lowers_gradient_error(w):
    # Controlled ablation (same kernels, D from O + Ores versus from O alone) at the pages' crop
    # sizes and head dimensions. dQ and dK are compared on 32 evenly spaced slices (a slice's dQ,
    # dK depend on that slice alone), dBias on 32 rows summed over every slice.
    import json
    import os

    import oracle

    x = wl.inputs_for(w)
    comp = run_cuda(x, residual=True)
    plain = run_cuda(x, residual=False)
    N = w.N
    sl = sorted(set(int(round(k * (N - 1) / 31)) for k in range(32)))
    sub = {k: (v[:, sl] if (v is not None and k in ("Q", "K", "V", "dO", "mask")) else v) for k, v in x.items()}
    want = oracle_full(sub)
    rows = [(0, h, j) for h in range(w.H) for j in range(0, N, N // 8)]
    want_rows = oracle.dbias_rows(x["Q"], x["K"], x["V"], x["bias"], x["mask"], x["dO"], rows)
    report = {}
    for k in ("dQ", "dK", "dBias"):
        if k == "dBias":
            gc = np.stack([f64(comp[k][b, h, j]) for (b, h, j) in rows])
            gp = np.stack([f64(plain[k][b, h, j]) for (b, h, j) in rows])
            ref = want_rows
        else:
            gc, gp, ref = f64(comp[k][:, sl]), f64(plain[k][:, sl]), want[k]
        ec, ep = rmse_rel(gc, ref), rmse_rel(gp, ref)
        # the gradients are returned in BF16: their error has a floor, the BF16 rounding of the exact
        # value, which no compensation removes; the residual acts on the error above it
        floor = rmse_rel(torch.from_numpy(np.asarray(ref)).to(torch.bfloat16).double().numpy(), ref)
        xc, xp = (max(e * e - floor * floor, 0.0) ** 0.5 for e in (ec, ep))
        report[k] = {"compensated": ec, "uncompensated": ep, "reduction": 1.0 - ec / ep, "bf16_floor": floor,
                     "reduction_above_floor": 1.0 - xc / xp if xp > 0 else 0.0}
        assert ec <= RMSE_REL_TOL, f"{w.name} {k}: compensated RMSE {ec}"
    print(f"residual ablation {w.name}:", json.dumps(report))
    out = os.environ.get("TRI_ATTN_ABLATION_LOG")
    if out:
        with open(out, "a") as f:
            f.write(json.dumps({"workload": w.name, **report}) + "\n")
    for k, r in report.items():
        assert r["reduction"] > 0.0, f"{w.name} {k}: residual compensation does not lower the error: {r}"
        assert r["reduction_above_floor"] >= MIN_GAIN_ABOVE_FLOOR, f"{w.name} {k}: {r}"


# The pages report 28-47 % lower dQ, dK and dBias RMSE from the residual at these crops. Here the
# gradients leave the kernels in BF16, whose own rounding (about 1.66e-3 relative RMSE) dominates
# their error; the residual must lower the total error on every crop and output, and the error
# above that rounding floor by at least 10 % (measured: 19.8 % at the least, crop 768 dK; up to
# 85 % at crop 384 dBias).
MIN_GAIN_ABOVE_FLOOR = 0.10


def test_residual_compensation_full_tensor_crop384():
    # the same ablation at crop 384 against the full oracle (every slice, the whole dBias)
    x = wl.inputs_for(wl.CROP384)
    want = oracle_full(x)
    comp = run_cuda(x, residual=True)
    plain = run_cuda(x, residual=False)
    for k in ("dQ", "dK", "dBias"):
        ec, ep = rmse_rel(f64(comp[k]), want[k]), rmse_rel(f64(plain[k]), want[k])
        assert ec < ep, f"{k}: compensated {ec} not below uncompensated {ep}"
    _compare_all(comp, want, "crop384")


def _sampled_check(x, slices, bias_rows, what, node=0):
    import oracle
    got = run_cuda(x, node=node)
    sub = {k: (v[:, slices] if (v is not None and k in ("Q", "K", "V", "dO", "mask")) else v)
           for k, v in x.items()}
    want = oracle_full(sub)
    for k in ("O", "dQ", "dK", "dV"):
        e = rmse_rel(f64(got[k][:, slices]), want[k])
        assert e <= RMSE_REL_TOL, f"{what}: {k} RMSE {e}"
        check_elementwise(f64(got[k][:, slices]), want[k], f"{what} {k}")
    check_lse(f64(got["LSE"][:, slices]), want["LSE"], what)
    rows = oracle.dbias_rows(x["Q"], x["K"], x["V"], x["bias"], x["mask"], x["dO"], bias_rows)
    gb = np.stack([f64(got["dBias"][b, h, j]) for (b, h, j) in bias_rows])
    e = rmse_rel(gb, rows)
    assert e <= RMSE_REL_TOL, f"{what}: dBias sampled-row RMSE {e}"
    check_elementwise(gb, rows, f"{what} dBias rows")
    return got


def _split_slices(w, node=0):
    """The sampled slices of a full-size case: first, middle and last, plus every slice that
    straddles one of the backward's cluster-range boundaries on this device."""
    from bwd_tri_attn_gb300 import binding as tb

    shape = tb.Shape(w.B, w.slices, w.N, w.H, w.d, 1.0 / w.d ** 0.5, node)
    extra, _ = boundary_slices(shape, w.slices)
    N = w.N
    return sorted(set([0, N // 3, N - 1] + extra))


FULL = [wl.CROP384, wl.CROP640_D16, wl.CROP640_D32, wl.CROP768]


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size_sampled(w):
    x = wl.inputs_for(w)
    N = w.N
    rows = [(0, h, j) for h in range(w.H) for j in (0, N // 2 + 1, N - 1)]
    _sampled_check(x, _split_slices(w), rows, w.name)


def test_ending_node_full_size():
    # the ending-node variant: the same op on the pair tensor with its two pair axes swapped
    x = wl.inputs_for(wl.CROP768)
    for k in ("Q", "K", "V", "dO"):
        x[k] = wl.ending_node(x[k])
    N = wl.CROP768.N
    _sampled_check(x, [1, N // 2, N - 2], [(0, 1, 5), (0, 3, N - 1), (0, 0, 400)], "ending_node")


def test_ending_node_in_place_full_size():
    # the ending node on the pair tensors as they are in memory (slices along the second pair
    # axis): no transposed copies
    x = wl.inputs_for(wl.CROP768)
    N = wl.CROP768.N
    slices = sorted(set([2, N // 2 + 3, N - 1] + _split_slices(wl.CROP768, node=1)))
    _sampled_check(x, slices, [(0, 2, 7), (0, 1, N - 1), (0, 3, 333)], "ending_node_in_place", node=1)


ENDING = [
    ("end_ragged_d32", dict(B=2, S=5, N=200, H=3, d=32, seed=31, mask=("random", 0.1))),
    ("end_ragged_d16", dict(B=1, S=9, N=77, H=2, d=16, seed=32, mask=("tail", 7))),
    ("end_tall_d32", dict(B=1, S=3, N=300, H=4, d=32, seed=33, mask=("zeros",))),
    ("end_wide_d16", dict(B=2, S=40, N=24, H=1, d=16, seed=34, mask=("none",))),
]


@pytest.mark.parametrize("name,cfg", ENDING, ids=[e[0] for e in ENDING])
def test_ending_node_in_place_full_oracle(name, cfg):
    x = wl.make_inputs(**cfg)
    got = run_cuda(x, node=1)
    want = oracle_full(x)
    _compare_all(got, want, name)
    # the same attention through the starting-node layout gives the same bits
    ref = run_cuda(x)
    for k in ("O", "LSE", "Ores", "dQ", "dK", "dV", "dBias"):
        assert torch.equal(got[k].view(torch.uint8), ref[k].view(torch.uint8)), f"{name}: {k} differs by layout"


def test_bitwise_determinism_five_calls():
    from bwd_tri_attn_gb300 import binding as tb
    x = wl.inputs_for(wl.CROP768)
    dx = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    ref = None
    for _ in range(5):
        O, LSE, Ores = tb.forward(dx["Q"], dx["K"], dx["V"], dx["bias"], dx["mask"])
        grads = tb.backward(dx["Q"], dx["K"], dx["V"], dx["bias"], dx["mask"], O, Ores, LSE, dx["dO"])
        outs = [O, LSE, Ores, *grads]
        torch.cuda.synchronize()
        if ref is None:
            ref = [t.clone() for t in outs]
        else:
            for a, b in zip(ref, outs):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert tb.tri_attn_device_status() == 0
