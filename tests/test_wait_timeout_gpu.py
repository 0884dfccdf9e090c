"""Failure detection on the GPU without a fault: a bounded wait that runs out.

tests/csrc/wait_timeout_probe.cu builds the attention kernels' wait helpers
(sync.cuh) into a one-CTA kernel whose first warp waits on an mbarrier that
nothing arrives on and whose second warp waits on another one. The first wait
must expire after the kernels' limit, raise the abort flag and write the
timeout status; the second must leave through the abort flag; the kernel must
return normally and the CUDA context must stay usable afterwards.
"""
import ctypes
import os
import subprocess
import time

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STATUS_TIMEOUT = 1  # kStatusTimeout in csrc/common.cuh, TRI_ATTN_ERR_TIMEOUT on the host side


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bwd_tri_attn_gb300 import _build
    out = os.path.join(_build.OBJDIR, "libwait_timeout_probe.so")
    os.makedirs(_build.OBJDIR, exist_ok=True)
    src = os.path.join(ROOT, "tests", "csrc", "wait_timeout_probe.cu")
    subprocess.run([_build.nvcc(), *_build.NVCC_FLAGS, "-shared", src, "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.wait_timeout_probe.argtypes = [ctypes.c_void_p] * 3
    lib.wait_timeout_probe.restype = ctypes.c_int
    lib.wait_limit_ns.restype = ctypes.c_ulonglong
    return lib


def test_wait_expires_and_kernel_returns(probe):
    limit = probe.wait_limit_ns()
    assert 0 < limit <= 5_000_000_000
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ok = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    ns = torch.zeros(2, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    rc = probe.wait_timeout_probe(status.data_ptr(), ok.data_ptr(), ns.data_ptr())
    wall = time.perf_counter() - t0
    assert rc == 0, f"probe kernel returned CUDA error {rc}"
    assert int(status.item()) == STATUS_TIMEOUT
    assert ok.tolist() == [0, 0]
    w0, w1 = (int(v) for v in ns.tolist())
    # warp 0 gave up at its own limit; warp 1 (started 0.1 s later) left through the abort flag,
    # well before its own limit would have expired
    assert limit <= w0 < limit + 500_000_000
    assert abs(w1 - w0) < 50_000_000
    assert wall < limit / 1e9 + 10
    # the context still works
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2
