"""Concurrent use of the library from several host threads.

The C ABI holds no per-call host state: tensor maps are built per call, and the
one-time per-device set-up (shared-memory attribute, residency queries) is
recorded in atomics. Two host threads that call forward + backward at the same
time, each on its own stream and its own workspace, must get exactly the
results of a single-threaded call. ctypes releases the GIL around each C call,
so the calls really overlap.
"""
import threading

import pytest
import torch

from bwd_tri_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bwd_tri_attn_gb300 import _build, binding
    _build.build()
    binding.load()


def _run(tb, x, node, stream):
    with torch.cuda.stream(stream):
        O, LSE, Ores = tb.forward(x["Q"], x["K"], x["V"], x["bias"], x["mask"], node=node, stream=stream)
        g = tb.backward(x["Q"], x["K"], x["V"], x["bias"], x["mask"], O, Ores, LSE, x["dO"], node=node,
                        stream=stream)
    stream.synchronize()
    return [O, LSE, Ores, *g]


def test_two_host_threads_match_single_thread():
    from bwd_tri_attn_gb300 import binding as tb

    cases = [(wl.make_inputs(B=1, S=40, N=384, H=4, d=32, seed=51, mask=("random", 0.05)), 0),
             (wl.make_inputs(B=2, S=24, N=200, H=2, d=16, seed=52, mask=("tail", 11)), 1)]
    dev = []
    for x, node in cases:
        d = {k: (None if v is None else v.cuda()) for k, v in x.items()}
        if node:
            d = {k: (v.transpose(1, 2).contiguous() if k in ("Q", "K", "V", "dO") else v) for k, v in d.items()}
        dev.append((d, node))
    ref = [_run(tb, d, node, torch.cuda.Stream()) for d, node in dev]
    for _ in range(3):
        out = [None, None]
        errs = []

        def worker(i):
            try:
                out[i] = _run(tb, dev[i][0], dev[i][1], torch.cuda.Stream())
            except Exception as e:  # reported below
                errs.append(e)

        ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert not errs, errs
        for i in range(2):
            for a, b in zip(ref[i], out[i]):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0


def _run_module(tb, x, H, d, node, stream):
    keys = ("z", "gamma", "beta", "W", "wb", "Wo")
    with torch.cuda.stream(stream):
        out, saved = tb.module_forward(*[x[k] for k in keys], x["mask"], H, d, node=node, stream=stream)
        g = tb.module_backward(*[x[k] for k in keys], x["mask"], saved, x["dout"], H, d, node=node, stream=stream)
    stream.synchronize()
    return [out, *g]


def test_two_host_threads_run_the_block_as_one_thread():
    """The triangle-attention block from two host threads at once, on two shapes that take different
    GEMM tile widths, LayerNorm templates and nodes (when no earlier call in the process has done
    so, their one-time per-device set-up runs inside the threads), bit for bit the single-threaded
    results."""
    from bwd_tri_attn_gb300 import binding as tb

    cases = [(wl.make_module_inputs(1, 56, 128, 4, 32, seed=61, mask=("tail", 3)), 4, 32, 0),
             (wl.make_module_inputs(2, 40, 256, 8, 16, seed=62, mask=("random", 0.1)), 8, 16, 1)]
    dev = [({k: (None if v is None else v.cuda()) for k, v in x.items()}, H, d, node) for x, H, d, node in cases]
    for _ in range(2):
        out = [None, None]
        errs = []

        def worker(i):
            try:
                x, H, d, node = dev[i]
                out[i] = _run_module(tb, x, H, d, node, torch.cuda.Stream())
            except Exception as e:  # reported below
                errs.append(e)

        ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert not errs, errs
        ref = [_run_module(tb, x, H, d, node, torch.cuda.Stream()) for x, H, d, node in dev]
        for i in range(2):
            for a, b in zip(ref[i], out[i]):
                assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
    torch.cuda.synchronize()
    assert tb.tri_attn_device_status() == 0
