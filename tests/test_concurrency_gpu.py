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
