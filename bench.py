"""Triangle-attention forward + backward throughput on GB300.

One step = one pass of the whole path (forward, D correction, main backward,
dBias reduction) over one batch of synthetic input of the named workload.
Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--node starting|ending]
                  [--impl ours|reference]

With N > 1 (torchrun, one process per GPU) every rank runs an independent
replica of the workload (the path has no cross-GPU exchange at this size):
weak scaling, the max over ranks of the timed region is used, and value is the
work of all ranks divided by that time. Run without torchrun, --gpus N > 1
starts itself under torch.distributed.run with N processes.

Timing: W untimed warm-up steps, then R windows of exactly K steps each, every
window bracketed by a barrier and a device synchronisation on both sides and
timed with CUDA events on the launching stream; the line reports the median
window (R >= 3, enough windows to fill about a second, so that the clock
sampler sees the GPU under load).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "triangle-attn fwd+bwd TFLOP/s at N=768,H=4,d=32 (1 GB300; % BF16 peak)"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 2**20

# Kernels each step enqueues, in order (the library's per-kernel event order).
KERNELS = ["fwd_vscale", "fwd", "bias_transpose", "bwd_prep", "bwd_main", "dbias_reduce"]
NFWD = 2  # kernels of tri_attn_fwd


# ncu summaries under profiles/ carry, per kernel, the DRAM bytes of one captured
# launch, the workload and activation size it ran on and a digest of the sources it was
# built from; traffic is reported only while the sources still match.
PROFILES = {"fwd": ("fwd_kernel_crop384_h4_d32.md", ["fwd.cu"]),
            "bwd_main": ("bwd_kernel_crop384_h4_d32.md", ["bwd.cu"])}
COMMON_SOURCES = ["common.cuh", "sm100.cuh", "sync.cuh", "tmap.cuh"]


def source_digest(own) -> str:
    """First 16 hex digits of the SHA-256 of a kernel's sources and the shared headers, with
    comments removed and whitespace collapsed: a change to the code renews it, a change to a
    comment does not."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in list(own) + COMMON_SOURCES:
        with open(os.path.join(ROOT, "bwd_tri_attn_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update((" ".join(src.split()) + "\n").encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, activation_elements: int):
    """(DRAM bytes per launch, how they were obtained) from the kernel's ncu summary: the captured
    launch's figure when it ran on a workload of this activation size, else scaled by activation
    size (every input of the square crops grows with S*N*H*d); (None, reason) when the summary is
    missing or the kernel's sources changed since it was taken."""
    name, own = PROFILES[kernel]
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
        digest = source_digest(own)
    except OSError:
        return None, "no ncu summary"
    fields = {}
    for line in text.splitlines():
        k, _, v = line.strip().partition(": ")
        if k in ("source_digest", "dram_bytes_per_launch", "activation_elements", "workload"):
            fields[k] = v.strip()
    if len(fields) != 4:
        return None, "ncu summary incomplete"
    if fields["source_digest"] != digest:
        return None, "kernel sources changed since the ncu capture"
    captured = int(fields["activation_elements"])
    bytes_ = int(fields["dram_bytes_per_launch"])
    if captured == activation_elements:
        return bytes_, f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one {fields['workload']} launch"
    return (bytes_ * activation_elements / captured,
            f"ncu DRAM bytes of one {fields['workload']} launch, scaled by activation size")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.file.name)
        return self.parse(rows)

    @staticmethod
    def parse(rows):
        """Median SM clock, max clock and the throttle reasons seen in nvidia-smi CSV rows."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the slowest rank's time); a no-op on one rank."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def bwd_unit_start(c: int, nc: int, w: int) -> int:
    """First (head, slice) pair of cluster c when the backward splits w pairs over nc clusters."""
    return c * w // nc


def bwd_cluster_of(x: int, nc: int, w: int) -> int:
    c = x * nc // w
    while c + 1 < nc and bwd_unit_start(c + 1, nc, w) <= x:
        c += 1
    while c > 0 and bwd_unit_start(c, nc, w) > x:
        c -= 1
    return c


def hbm_algorithmic_bytes(B, S, N, H, d, nc):
    """Bytes each HBM-bound kernel must move at least once (reads + writes), per launch."""
    nx = B * S * N * H * d
    NP = (N + 127) // 128 * 128
    njt = NP // 128
    w = B * H * S
    slots = sum(bwd_cluster_of(hd * S + S - 1, nc, w) - bwd_cluster_of(hd * S, nc, w) + 1 for hd in range(B * H))
    return {
        "fwd_vscale": 2 * nx + 4 * B * S * H * njt,                        # V in; one int per work unit out
        "bias_transpose": 2 * B * H * N * N + 2 * B * H * NP * NP,         # bias in; padded transpose out
        "bwd_prep": 6 * 2 * nx + 4 * B * S * H * N + 16 * B * S * H,      # dO, O, Ores, Q, K, V in; D, scales out
        "dbias_reduce": 4 * slots * N * NP + 2 * B * H * N * N,            # FP32 partial slots in; BF16 dBias out
    }


def hbm_report(kernel_ms, B, S, N, H, d, nc, peak_gbs):
    out = {}
    for k, nbytes in hbm_algorithmic_bytes(B, S, N, H, d, nc).items():
        gbs = nbytes / (kernel_ms[k] * 1e-3) / 1e9
        out[k] = {"bytes": nbytes, "ms": kernel_ms[k], "gbs": gbs, "frac": gbs / peak_gbs}
    return out


def job_throughput(world: int, flops_per_step: float, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs the same step on its own data (weak scaling), and the
    job's step time is the slowest rank's."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


def cpu_oracle_sample(w, slices: int, nthreads: int = 0):
    """Times the FP64 oracle's forward + backward on `slices` slices of the workload."""
    import oracle
    from bwd_tri_attn_gb300 import workloads as wl

    x = wl.inputs_for(w, slices=slices)
    args = [oracle._f64(x[k]) for k in ("Q", "K", "V", "bias", "mask", "dO")]
    cores = oracle.num_threads(nthreads)
    t0 = time.perf_counter()
    oracle.fwd(*args[:5], nthreads=nthreads)
    oracle.bwd(*args, nthreads=nthreads)
    dt = time.perf_counter() - t0
    flops = 14.0 * w.B * slices * w.H * w.N * w.N * w.d
    return flops / dt / 1e12, dt, cores


def config_of(w, node: str) -> dict:
    """The workload description both arms print (identical, so that their lines compare)."""
    return {"workload": w.name, "B": w.B, "S": w.slices, "N": w.N, "H": w.H, "d": w.d, "node": node,
            "mask": list(w.mask), "flops_per_step": w.flops()}


def run_reference(args, w):
    """Reference arm: the FP64 oracle on the host cores, one bounded sample per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    slices = args.ref_slices
    for _ in range(args.warmup):
        cpu_oracle_sample(w, slices)
    times, cores = [], 1
    for _ in range(args.steps):
        _, dt, cores = cpu_oracle_sample(w, slices)
        times.append(dt)
    t = sum(times)
    flops = 14.0 * w.B * slices * w.H * w.N * w.N * w.d
    value = flops * args.steps / t / 1e12
    sample = f"{slices} of {w.slices} slices (all {w.H} heads, full N={w.N}) per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, args.node),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# Triangle multiplicative update, measured beside the attention (same step discipline):
# kernels per fwd+bwd step in the library's event order, per layout of the projections.
MUL_KERNELS = {0: ["mul_gate", "mul_gemm_x", "mul_gemm_da", "mul_gemm_db", "mul_gate_bwd"],
               1: ["mul_gate", "mul_gemm_x", "mul_gemm_da_gate", "mul_gemm_db_gate"]}
MUL_NFWD = 2


def mul_roofline(kernel_ms, B, N, C, peaks):
    """Per-kernel roofline of the triangle multiplication: the three contractions against the BF16
    tensor peak (2 B C N^3 FLOPs each) and all kernels against HBM. Algorithmic bytes per element of
    one [B, N, N, C] tensor: gating reads P, G of both operands and writes both gated operands
    (12 B); the X contraction reads A, Bm and writes X (6 B); in the pair layout the dA and dB
    contractions read two BF16 operands and write FP32 (8 B) and the gating gradient reads dA, dB,
    P, G of both operands and writes four BF16 gradients (24 B); in the channel-major layout each
    backward contraction reads two operands, P and G, and writes dP and dG (12 B)."""
    E = B * N * N * C
    flops = 2.0 * B * C * float(N) ** 3
    bytes_of = {"mul_gate": 12 * E, "mul_gemm_x": 6 * E, "mul_gemm_da": 8 * E, "mul_gemm_db": 8 * E,
                "mul_gate_bwd": 24 * E, "mul_gemm_da_gate": 12 * E, "mul_gemm_db_gate": 12 * E}
    out = {}
    for k, ms in kernel_ms.items():
        gbs = bytes_of[k] / (ms * 1e-3) / 1e9
        r = {"ms": ms, "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"], "bytes": bytes_of[k]}
        if "gemm" in k:
            tf = flops / (ms * 1e-3) / 1e12
            r.update({"tflops": tf, "tensor_frac": tf / peaks["bf16_tflops"]})
        out[k] = r
    return out


def run_trimul(dev, stream, steps, incoming=False, layout=1, mw=None):
    """Times the triangle multiplicative update (fwd + bwd); default workload crop 768, 128 channels."""
    import torch

    from bwd_tri_attn_gb300 import binding as tb
    from bwd_tri_attn_gb300 import workloads as wl

    mw = mw or wl.MUL_CROP768
    x = {k: v.to(dev) for k, v in wl.mul_inputs_for(mw).items()}
    if layout == tb.LAYOUT_CHANNEL_MAJOR:
        x = {k: (v.permute(0, 3, 1, 2).contiguous() if k != "dX" else v) for k, v in x.items()}
    shape = tb.mul_shape_of(x["Pa"], incoming, layout)
    B, N, C = shape.B, shape.N, shape.C
    A, Bm, X = (torch.empty((B, C, N, N), dtype=torch.bfloat16, device=dev) for _ in range(3))
    grads = [torch.empty_like(x["Pa"]) for _ in range(4)]
    ws = torch.empty(max(16, tb.tri_mul_bwd_workspace_size(shape)), dtype=torch.uint8, device=dev)
    names = MUL_KERNELS[layout]

    def step(marks=None):
        if marks:
            tb.tri_attn_set_timing_events(marks[:MUL_NFWD])
        tb.tri_mul_fwd(shape, x["Pa"], x["Ga"], x["Pb"], x["Gb"], A, Bm, X, stream)
        if marks:
            tb.tri_attn_set_timing_events(marks[MUL_NFWD:])
        tb.tri_mul_bwd(shape, x["Pa"], x["Ga"], x["Pb"], x["Gb"], A, Bm, x["dX"], *grads, ws, stream)

    for _ in range(3):
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    marks = [[torch.cuda.Event(enable_timing=True) for _ in names] for _ in range(steps)]
    for e in starts + [m for ms in marks for m in ms]:
        e.record(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for k in range(steps):
        starts[k].record(stream)
        step(marks[k])
    t1.record(stream)
    tb.tri_attn_set_timing_events(None)
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
    per = {n: 0.0 for n in names}
    for k in range(steps):
        chain = [starts[k]] + marks[k]
        for n, (a, b) in enumerate(zip(chain[:-1], chain[1:])):
            per[names[n]] += a.elapsed_time(b) / steps
    ms = t0.elapsed_time(t1) / steps
    peaks = load_peaks()
    return {"workload": mw.name, "direction": "incoming" if incoming else "outgoing",
            "layout": "channel-major" if layout == tb.LAYOUT_CHANNEL_MAJOR else "pair",
            "B": B, "N": N, "C": C, "ms_per_step": ms, "tflops": 3 * mw.flops() / (ms * 1e-3) / 1e12,
            "flops_per_step": 3 * mw.flops(), "steps": steps,
            "l2": f"inputs and operands larger than L2 (each [B,N,N,C] tensor is {2 * B * N * N * C / 1e6:.0f} MB; "
                  "four projections per step), no flush",
            "kernels": mul_roofline(per, B, N, C, peaks), "gpu_launches": steps * len(names)}


def run_trimul_only(args):
    """``--trimul-only``: the triangle multiplication sub-line alone (one GPU), for profiling."""
    import torch

    from bwd_tri_attn_gb300 import _build
    from bwd_tri_attn_gb300 import binding as tb
    from bwd_tri_attn_gb300 import workloads as wl

    _build.build()
    tb.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    mw = wl.MUL_ALL[args.mul_workload]
    out = [run_trimul(dev, stream, args.steps, incoming=inc, layout=lay, mw=mw)
           for lay in (tb.LAYOUT_CHANNEL_MAJOR, tb.LAYOUT_PAIR) for inc in (False, True)]
    print(json.dumps({"trimul": out}))


MOD_KERNELS = ["mod_ln_fwd", "mod_proj_gemm", "fwd_vscale", "fwd", "mod_gate", "mod_out_gemm",
               "mod_dgo_gemm", "mod_dwo_gemm", "mod_dwo_reduce", "bias_transpose", "bwd_prep", "bwd_main",
               "dbias_reduce", "mod_dzt_gemm", "mod_ln_bwd", "mod_ln_reduce", "mod_dw_gemm", "mod_dw_reduce"]
MOD_NFWD = 6


def mod_roofline(kernel_ms, B, N, c, H, d, peaks):
    """Per-kernel figures of the triangle-attention block's own kernels (the attention's are reported
    by the main line). M = B N^2 pair positions, hd = H d; algorithmic bytes (each tensor read or
    written once) and GEMM FLOPs:
      LayerNorm forward: z in, zt out (2 M c each), mean and 1/std (8 M), pair bias (2 M H);
      input projections: zt in (2 M c), q, k, v, gl out (8 M hd); 2 M c 4hd FLOPs;
      gate: gl and O in, go out (6 M hd); output projection: go in (2 M hd), out (2 M c), 2 M hd c FLOPs;
      dgo with the gate gradient: dout (2 M c), O and gl in, dO and dgl out (8 M hd), 2 M c hd FLOPs;
      dWo partials: dout and go in (2 M c + 2 M hd), 2 M c hd FLOPs;
      dzt: dq, dk, dv, dgl in (8 M hd), dzt out in FP32 (4 M c), 2 M 4hd c FLOPs;
      LayerNorm backward: dzt (4 M c), z, zt (4 M c), statistics (8 M), dbias (2 M H) in, dz out (2 M c);
      dW partials: dq, dk, dv, dgl and zt in (8 M hd + 2 M c), 2 M 4hd c FLOPs."""
    M = B * N * N
    hd = H * d
    spec = {"mod_ln_fwd": (4 * M * c + 8 * M + 2 * M * H, 0),
            "mod_proj_gemm": (2 * M * c + 8 * M * hd, 2.0 * M * c * 4 * hd),
            "mod_gate": (6 * M * hd, 0),
            "mod_out_gemm": (2 * M * hd + 2 * M * c, 2.0 * M * hd * c),
            "mod_dgo_gemm": (2 * M * c + 8 * M * hd, 2.0 * M * c * hd),
            "mod_dwo_gemm": (2 * M * c + 2 * M * hd, 2.0 * M * c * hd),
            "mod_dzt_gemm": (8 * M * hd + 4 * M * c, 2.0 * M * 4 * hd * c),
            "mod_ln_bwd": (10 * M * c + 8 * M + 2 * M * H, 0),
            "mod_dw_gemm": (8 * M * hd + 2 * M * c, 2.0 * M * 4 * hd * c)}
    out = {}
    for k, (nbytes, flops) in spec.items():
        ms = kernel_ms[k]
        gbs = nbytes / (ms * 1e-3) / 1e9
        r = {"ms": ms, "bytes": nbytes, "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"]}
        if flops:
            tf = flops / (ms * 1e-3) / 1e12
            r.update({"tflops": tf, "tensor_frac": tf / peaks["bf16_tflops"]})
        out[k] = r
    return out


def run_module(dev, stream, steps, mw=None):
    """Times the triangle-attention block (LayerNorm, projections, attention, gate, output projection),
    forward and backward; default workload crop 768, 128 pair channels, H = 4, d = 32."""
    import torch

    from bwd_tri_attn_gb300 import binding as tb
    from bwd_tri_attn_gb300 import workloads as wl

    mw = mw or wl.MOD_CROP768
    x = {k: (None if v is None else v.to(dev)) for k, v in wl.module_inputs_for(mw).items()}
    args = [x[k] for k in ("z", "gamma", "beta", "W", "wb", "Wo")]
    shape = tb.module_shape_of(x["z"], mw.H, mw.d, mw.node)
    saved = torch.empty(tb.tri_module_saved_size(shape), dtype=torch.uint8, device=dev)
    ws = torch.empty(tb.tri_module_bwd_workspace_size(shape), dtype=torch.uint8, device=dev)
    out = torch.empty_like(x["z"])
    f32 = dict(dtype=torch.float32, device=dev)
    grads = [torch.empty_like(x["z"]), torch.empty(mw.c, **f32), torch.empty(mw.c, **f32),
             torch.empty(x["W"].shape, **f32), torch.empty(x["wb"].shape, **f32), torch.empty(x["Wo"].shape, **f32)]

    def step(marks=None):
        if marks:
            tb.tri_attn_set_timing_events(marks[:MOD_NFWD])
        tb.tri_module_fwd(shape, *args, x["mask"], out, saved, stream)
        if marks:
            tb.tri_attn_set_timing_events(marks[MOD_NFWD:])
        tb.tri_module_bwd(shape, *args, x["mask"], saved, x["dout"], *grads, ws, stream)

    for _ in range(3):
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    marks = [[torch.cuda.Event(enable_timing=True) for _ in MOD_KERNELS] for _ in range(steps)]
    for e in starts + [m for ms in marks for m in ms]:
        e.record(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for k in range(steps):
        starts[k].record(stream)
        step(marks[k])
    t1.record(stream)
    tb.tri_attn_set_timing_events(None)
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
    per = {n: 0.0 for n in MOD_KERNELS}
    for k in range(steps):
        chain = [starts[k]] + marks[k]
        for n, (a, b) in enumerate(zip(chain[:-1], chain[1:])):
            per[MOD_KERNELS[n]] += a.elapsed_time(b) / steps
    ms = t0.elapsed_time(t1) / steps
    peaks = load_peaks()
    M = mw.B * mw.N * mw.N
    attn = ("fwd_vscale", "fwd", "bias_transpose", "bwd_prep", "bwd_main", "dbias_reduce")
    around = sum(v for k, v in per.items() if k not in attn)
    return {"workload": mw.name, "B": mw.B, "N": mw.N, "c": mw.c, "H": mw.H, "d": mw.d,
            "node": "starting" if mw.node == 0 else "ending", "ms_per_step": ms,
            "tflops": mw.flops() / (ms * 1e-3) / 1e12, "flops_per_step": mw.flops(), "steps": steps,
            "attention_ms": sum(per[k] for k in attn), "around_attention_ms": around,
            "l2": f"inputs and activations larger than L2 (z alone is {2 * M * mw.c / 1e6:.0f} MB), no flush",
            "kernel_ms": per, "kernels": mod_roofline(per, mw.B, mw.N, mw.c, mw.H, mw.d, peaks),
            "gpu_launches": steps * len(MOD_KERNELS)}


def run_module_only(args):
    """``--module-only``: the triangle-attention block sub-line alone (one GPU), for profiling."""
    import torch

    from bwd_tri_attn_gb300 import _build
    from bwd_tri_attn_gb300 import binding as tb
    from bwd_tri_attn_gb300 import workloads as wl

    _build.build()
    tb.load()
    dev = torch.device("cuda", 0)
    print(json.dumps({"module": run_module(dev, torch.cuda.current_stream(), args.steps,
                                           wl.MOD_ALL[args.mod_workload])}))


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from bwd_tri_attn_gb300 import binding as tb
    from bwd_tri_attn_gb300 import workloads as wl
    from bwd_tri_attn_gb300 import _build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    tb.load()

    x = wl.inputs_for(w)
    node = tb.NODE_ENDING if args.node == "ending" else tb.NODE_STARTING
    if node == tb.NODE_ENDING:  # the ending node's pair tensors hold the slices along the second pair axis
        x = {k: (v.transpose(1, 2).contiguous() if k in ("Q", "K", "V", "dO") else v) for k, v in x.items()}
    d = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    shape = tb.shape_of(d["Q"], node=node)
    B, S, N, H, hd = shape.B, shape.S, shape.N, shape.H, shape.d
    O = torch.empty_like(d["Q"])
    Ores = torch.empty_like(d["Q"])
    LSE = torch.empty((B, S, H, N), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(O), torch.empty_like(O), torch.empty_like(O)
    dBias = torch.empty_like(d["bias"])
    ws = tb.workspace_for(shape, dev)
    stream = torch.cuda.current_stream()

    def step():
        tb.tri_attn_fwd(shape, d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, LSE, Ores, stream)
        tb.tri_attn_bwd(shape, d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, Ores, LSE, d["dO"], dQ, dK, dV,
                        dBias, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # per-kernel events: one after each kernel of the step (KERNELS order), after a start event
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS))] for _ in range(K)]
    for e in starts + [m for ms in marks for m in ms]:
        e.record(stream)  # materialise the events before handing their handles over
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    per_kernel = {n: [] for n in KERNELS}

    def window():
        """Exactly K timed steps, bracketed by a barrier and a synchronisation on both sides;
        returns the slowest rank's elapsed milliseconds."""
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for k in range(K):
            starts[k].record(stream)
            tb.tri_attn_set_timing_events(marks[k][:NFWD])
            tb.tri_attn_fwd(shape, d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, LSE, Ores, stream)
            tb.tri_attn_set_timing_events(marks[k][NFWD:])
            tb.tri_attn_bwd(shape, d["Q"], d["K"], d["V"], d["bias"], d["mask"], O, Ores, LSE, d["dO"], dQ, dK,
                            dV, dBias, ws, stream)
        t_end.record(stream)
        tb.tri_attn_set_timing_events(None)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        for k in range(K):
            chain = [starts[k]] + marks[k]
            for n, (a, b) in enumerate(zip(chain[:-1], chain[1:])):
                per_kernel[KERNELS[n]].append(a.elapsed_time(b))
        return max_over_ranks(t_start.elapsed_time(t_end), world, dev)

    with ClockSampler(torch.cuda.current_device()) as clocks:
        windows = [window()]
        nwin = args.windows or max(3, min(50, int(1000.0 / max(windows[0], 1e-3)) + 1))
        nwin = max_over_ranks(nwin, world, dev)  # every rank runs the same number of windows
        while len(windows) < nwin:
            windows.append(window())
    elapsed_ms = statistics.median(windows)
    assert tb.tri_attn_device_status() == 0
    kernel_ms = {n: sum(v) / len(v) for n, v in per_kernel.items()}

    flops = w.flops()
    ms_per_step = elapsed_ms / K
    value = job_throughput(world, flops, ms_per_step)
    peaks = load_peaks()

    # roofline of the dominant kernel (tensor-bound contraction; FP16 operands run at the BF16 rate)
    flops_of = {"fwd": 4.0 * B * S * H * N * N * hd, "bwd_main": 10.0 * B * S * H * N * N * hd}
    dom = max(("fwd", "bwd_main"), key=lambda n: kernel_ms[n])
    achieved = flops_of[dom] / (kernel_ms[dom] * 1e-3) / 1e12
    traffic, traffic_source = profiled_traffic(dom, B * S * N * H * hd)
    roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": traffic, "traffic_source": traffic_source,
                "peak_source": f"{peaks['source']} bf16 dense burst"}

    # HBM-bound kernels: algorithmic bytes / time
    nc, _ = tb.tri_attn_bwd_split(shape)
    hbm = hbm_report(kernel_ms, B, S, N, H, hd, nc, peaks["hbm_gbs"])

    # end to end through the public API: pinned host inputs -> device -> fwd+bwd -> gradients back to host.
    # Every step copies its own inputs in and its four gradients out inside the timed region. The
    # copies are pipelined like a prefetching data loader: two device buffer sets, the host->device
    # copy of step k+1 and the device->host copy of step k-1 on their own streams while step k runs.
    e2e = None
    if not args.no_e2e:
        host_in = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dQ, dK, dV, dBias)]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values() if v is not None)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        sets = []
        for _ in range(2):
            din = {k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in x.items()}
            dout = [torch.empty_like(t) for t in (dQ, dK, dV, dBias)]
            fo = (torch.empty_like(O), torch.empty_like(Ores), torch.empty_like(LSE))
            sets.append((din, dout, fo, tb.workspace_for(shape, dev)))
        # one copy stream per large tensor, so that the copies of a step can run on several copy
        # engines at once
        NCS = 4
        s_in = [torch.cuda.Stream(device=dev) for _ in range(NCS)]
        s_out = [torch.cuda.Stream(device=dev) for _ in range(NCS)]
        in_items = [(kname, v) for kname, v in host_in.items() if v is not None]
        in_items.sort(key=lambda kv: -kv[1].numel() * kv[1].element_size())

        def e2e_run(n):
            """n pipelined steps; returns the events that bracket them."""
            ev_comp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [[] for _ in range(n)]
            e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e_start.record(stream)
            for s_ in s_in + s_out:
                s_.wait_event(e_start)
            for k in range(n):
                din, dout, (o_, ores_, lse_), ws_ = sets[k % 2]
                for j, (kname, v) in enumerate(in_items):
                    s_ = s_in[j % NCS]
                    with torch.cuda.stream(s_):
                        if k >= 2 and j < NCS:
                            s_.wait_event(ev_comp[k - 2])  # step k-2 no longer reads this input set
                        din[kname].copy_(v, non_blocking=True)
                for s_ in s_in:
                    e = torch.cuda.Event()
                    e.record(s_)
                    stream.wait_event(e)
                if k >= 2:
                    for e in ev_out[k - 2]:  # step k-2's gradients have left this output set
                        stream.wait_event(e)
                tb.tri_attn_fwd(shape, din["Q"], din["K"], din["V"], din["bias"], din["mask"], o_, lse_, ores_, stream)
                tb.tri_attn_bwd(shape, din["Q"], din["K"], din["V"], din["bias"], din["mask"], o_, ores_, lse_, din["dO"],
                                dout[0], dout[1], dout[2], dout[3], ws_, stream)
                ev_comp[k].record(stream)
                for j, (src, dst) in enumerate(zip(dout, host_out)):
                    s_ = s_out[j % NCS]
                    with torch.cuda.stream(s_):
                        s_.wait_event(ev_comp[k])
                        dst.copy_(src, non_blocking=True)
                        e = torch.cuda.Event()
                        e.record(s_)
                        ev_out[k].append(e)
            for e in ev_out[n - 1]:
                stream.wait_event(e)
            e_end.record(stream)
            return e_start, e_end

        e2e_run(2)
        torch.cuda.synchronize()
        # three windows of ke pipelined steps (as many as the device-side windows, at least 40), each
        # bracketed by a barrier and a synchronisation; the median window is reported. Every window
        # contains the pipeline's fill (the first step's input copy, not overlapped) and drain (the
        # last step's gradient copy), about 5 ms at crop 768, which a long training run amortises.
        ke = max(K, 40)
        e_windows = []
        for _ in range(3):
            if world > 1:
                dist.barrier()
            e0, e1 = e2e_run(ke)
            torch.cuda.synchronize()
            e_windows.append(max_over_ranks(e0.elapsed_time(e1) / ke, world, dev))
        ems = statistics.median(e_windows)
        assert tb.tri_attn_device_status() == 0
        e2e = {"value": job_throughput(world, flops, ems), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems, "steps": ke, "window_ms_per_step": e_windows,
               "reported": "median of 3 windows",
               "pipelined": "two device buffer sets; H2D of step k+1 and D2H of step k-1 overlap step k; "
                            "one copy stream per large tensor"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, cores = cpu_oracle_sample(w, args.cpu_slices)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "seconds": dt,
               "sample": f"{args.cpu_slices} of {w.slices} slices (all {w.H} heads, full N={w.N}), fwd+bwd"}

    mul = None
    if not args.no_trimul:
        mw = wl.MUL_ALL[args.mul_workload]
        mul = [run_trimul(dev, stream, max(3, min(K, 20)), layout=lay, mw=mw)
               for lay in (tb.LAYOUT_CHANNEL_MAJOR, tb.LAYOUT_PAIR)]

    mod = None
    if not args.no_module:
        mod = run_module(dev, stream, max(3, min(K, 20)), wl.MOD_ALL[args.mod_workload])

    in_bytes = sum(v.numel() * v.element_size() for v in x.values() if v is not None)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, args.node),
            "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB of inputs vs {L2_BYTES / 1e6:.0f} MB L2), no flush",
            "operands": "BF16 in/out, FP16 tensor-core operands (power-of-two scaled per (batch, slice, head)), "
                        "FP32 accumulation",
            "timing": {"windows": len(windows), "steps_per_window": K, "window_ms": windows,
                       "reported": "median window"},
            "pct_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "pct_bf16_peak_sustained": 100.0 * value / world / peaks["bf16_tflops_sustained"],
            # the same step counted without the backward's P recompute (12 instead of 14 x B S H N^2 d)
            "value_12x_count": value * 12.0 / 14.0,
            "kernel_ms": kernel_ms, "hbm": hbm, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": K * len(KERNELS), "clocks": clocks.summary(), "trimul": mul, "module": mod,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    from bwd_tri_attn_gb300 import workloads as wl

    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.CROP768.name, choices=sorted(wl.ALL))
    ap.add_argument("--node", choices=["starting", "ending"], default="starting",
                    help="which pair axis holds the slices (the ending node reads the pair tensors in place)")
    ap.add_argument("--cpu-slices", type=int, default=384,
                    help="slices in the timed CPU oracle sample (about 10 s of host work at crop 768)")
    ap.add_argument("--ref-slices", type=int, default=4, help="slices per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-trimul", action="store_true", help="skip the triangle multiplication sub-line")
    ap.add_argument("--trimul-only", action="store_true",
                    help="time only the triangle multiplication (both layouts, both directions); one JSON line")
    ap.add_argument("--mul-workload", default=wl.MUL_CROP768.name, choices=sorted(wl.MUL_ALL))
    ap.add_argument("--no-module", action="store_true", help="skip the triangle-attention block sub-line")
    ap.add_argument("--module-only", action="store_true",
                    help="time only the triangle-attention block (forward and backward); one JSON line")
    ap.add_argument("--mod-workload", default=wl.MOD_CROP768.name, choices=sorted(wl.MOD_ALL))
    ap.add_argument("--windows", type=int, default=0,
                    help="timed windows of --steps steps (0: enough to fill about a second, at least 3)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "0"))
    if world == 0 and args.gpus > 1:
        # one process per GPU: start this script under torch.distributed.run
        import socket
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))
    if world and world != args.gpus:
        ap.error(f"--gpus {args.gpus} disagrees with WORLD_SIZE={world}")
    w = wl.ALL[args.workload]
    if args.trimul_only:
        run_trimul_only(args)
        return
    if args.module_only:
        run_module_only(args)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
