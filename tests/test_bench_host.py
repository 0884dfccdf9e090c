"""Host-side logic of bench.py, on CPU: the multi-rank aggregation (world size 2 over
gloo), the whole-job throughput, the reference arm's rank handling, the clock-record
parsing, the measured-peak lookup and the profile-digest check behind roofline.traffic.
"""
import hashlib
import json
import re
import os
import shutil
import socket
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's step time; the job is as slow as its slowest rank
        ms = 3.0 + 1.5 * rank
        slowest = bench.max_over_ranks(ms, world)
        value = bench.job_throughput(world, 0.8117e12, slowest)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["slowest"] == pytest.approx(4.5)
        # two replicas, each 0.8117 TFLOP per 4.5 ms step
        assert r["value"] == pytest.approx(2 * 0.8117e12 / 4.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_throughput(1, 1e12, 1000.0) == pytest.approx(1.0)


def test_reference_arm_only_rank_zero_works(monkeypatch, capsys):
    from bwd_tri_attn_gb300 import workloads as wl

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "cpu_oracle_sample", lambda *a, **k: called.append(a) or (1.0, 1.0, 1))
    args = types.SimpleNamespace(ref_slices=1, warmup=3, steps=2)
    bench.run_reference(args, wl.CROP768)
    assert called == [] and capsys.readouterr().out == ""


def test_clock_rows_parsing():
    rows = [
        "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1965, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1201.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 1201.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "short row",
    ]
    got = bench.ClockSampler.parse([r.split(",") for r in rows])
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0 and got["samples"] == 3
    assert got["reasons"] == ["sw_power_cap"]


def test_peaks_measured_then_fallback(monkeypatch, tmp_path):
    p = bench.load_peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert p["source"] == "measured" and p["bf16_tflops"] > 0
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks()["source"] == "fallback"


def test_traffic_reported_only_for_matching_sources(monkeypatch, tmp_path):
    src = os.path.join(ROOT, "bwd_tri_attn_gb300", "csrc")
    csrc = tmp_path / "bwd_tri_attn_gb300" / "csrc"
    shutil.copytree(src, csrc)
    (tmp_path / "profiles").mkdir()
    h = hashlib.sha256()
    for f in ["fwd.cu"] + bench.COMMON_SOURCES:
        code = re.sub(r"//[^\n]*", " ", re.sub(r"/\*.*?\*/", " ", (csrc / f).read_text(), flags=re.S))
        h.update((" ".join(code.split()) + "\n").encode())
    (tmp_path / "profiles" / "fwd_kernel_crop384_h4_d32.md").write_text(
        f"    source_digest: {h.hexdigest()[:16]}\n    workload: tiny\n    dram_bytes_per_launch: 1000\n"
        "    activation_elements: 10\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the captured launch's own figure at its size, scaled to another activation size
    assert bench.profiled_traffic("fwd", 10)[0] == 1000
    assert "one tiny launch" in bench.profiled_traffic("fwd", 10)[1]
    assert bench.profiled_traffic("fwd", 40)[0] == pytest.approx(4000.0)
    assert "scaled" in bench.profiled_traffic("fwd", 40)[1]
    # a comment or blank line added to a source leaves the code, and the figure, as it was
    with open(csrc / "common.cuh", "a") as f:
        f.write("\n// a remark\n/* and a block\n   comment */\n\n")
    assert bench.profiled_traffic("fwd", 10)[0] == 1000
    # a changed line of code invalidates it
    with open(csrc / "fwd.cu", "a") as f:
        f.write("\nstatic const int unused_probe = 0;\n")
    assert bench.profiled_traffic("fwd", 40)[0] is None
    # a missing summary reports nothing
    assert bench.profiled_traffic("bwd_main", 40)[0] is None
