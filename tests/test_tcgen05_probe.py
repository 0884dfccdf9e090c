"""Unit check of the tcgen05 / TMA operand layouts the attention kernels use.

A one-CTA probe (tests/csrc/tcgen05_probe.cu) computes S = A B^T (BF16,
K-major, TMA-swizzled), O = P V (P: FP16 A operand in TMEM, V: FP16 MN-major)
and O2 = X^T V (X: FP16 MN-major SW128 tile written by threads) and the
results are compared with host matmuls.
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from bwd_tri_attn_gb300 import _build
    out = os.path.join(_build.OBJDIR, "libtcgen05_probe.so")
    os.makedirs(_build.OBJDIR, exist_ok=True)
    src = os.path.join(ROOT, "tests", "csrc", "tcgen05_probe.cu")
    subprocess.run([_build.nvcc(), *_build.NVCC_FLAGS, "-shared", src, "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.tcgen05_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_float] + [ctypes.c_void_p] * 4
    lib.tcgen05_probe.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("hd", [16, 32])
def test_operand_layouts(probe, hd):
    g = torch.Generator().manual_seed(hd)
    A = torch.randn(128, hd, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(128, hd, generator=g).to(torch.bfloat16).cuda()
    V = torch.randn(128, hd, generator=g).to(torch.bfloat16).cuda()
    S = torch.empty(128, 128, device="cuda")
    O = torch.empty(128, hd, device="cuda")
    O2 = torch.empty(128, hd, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xscale = 0.125
    rc = probe.tcgen05_probe(A.data_ptr(), B.data_ptr(), V.data_ptr(), hd, xscale, S.data_ptr(), O.data_ptr(),
                             O2.data_ptr(), err.data_ptr())
    assert rc == 0 and int(err.item()) == 0
    S_ref = A.double() @ B.double().T
    torch.testing.assert_close(S.double(), S_ref, rtol=1e-5, atol=1e-5)
    P = (S * xscale).half().double()
    V16 = V.half().double()
    torch.testing.assert_close(O.double(), P @ V16, rtol=1e-4, atol=1e-4)
    torch.testing.assert_close(O2.double(), P.T @ V16, rtol=1e-4, atol=1e-4)
