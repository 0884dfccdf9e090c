"""Host-side checks of the C ABI (no GPU needed, no compute launched).

The library is built and loaded, every function declared in include/*.h must
be exported, and argument validation must reject bad calls on the host with
the documented codes before anything is enqueued.
"""
import ctypes
import glob
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bwd_tri_attn_gb300 import _build, binding
    _build.build()
    return binding.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(?:int|size_t|const char\s*\*|void)\s*\*?\s*(tri_(?:attn|mul|module)_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def _has_device():
    import torch
    return torch.cuda.is_available()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"tri_attn_fwd", "tri_attn_bwd", "tri_attn_bwd_workspace_size", "tri_attn_strerror",
            "tri_attn_device_status", "tri_attn_set_timing_events", "tri_attn_bwd_split",
            "tri_attn_bwd_static", "tri_mul_fwd", "tri_mul_bwd", "tri_mul_bwd_workspace_size", "tri_module_fwd",
            "tri_module_bwd", "tri_module_saved_size", "tri_module_bwd_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_strerror_covers_codes(lib):
    from bwd_tri_attn_gb300 import binding
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = binding.strerror(code)
        assert s and s != "unknown error code"
    assert binding.strerror(-99) == "unknown error code"


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced: validation fails first


def _fwd(lib, shape, **ptrs):
    from bwd_tri_attn_gb300.binding import Shape
    names = ["Q", "K", "V", "bias", "mask", "O", "LSE", "Ores"]
    args = [ctypes.c_void_p(ptrs.get(n, FAKE)) for n in names]
    return lib.tri_attn_fwd(Shape(*shape), *args, None)


def _bwd(lib, shape, ws_bytes, **ptrs):
    from bwd_tri_attn_gb300.binding import Shape
    names = ["Q", "K", "V", "bias", "mask", "O", "Ores", "LSE", "dO", "dQ", "dK", "dV", "dBias", "ws"]
    args = [ctypes.c_void_p(ptrs.get(n, FAKE)) for n in names]
    return lib.tri_attn_bwd(Shape(*shape), *args, ctypes.c_size_t(ws_bytes), None)


GOOD = (1, 4, 64, 2, 32, 0.17677669)


@pytest.mark.parametrize("shape,code", [
    ((0, 4, 64, 2, 32, 0.1), -1),          # empty batch
    ((1, 0, 64, 2, 32, 0.1), -1),          # no slices
    ((1, 4, 0, 2, 32, 0.1), -1),           # no positions
    ((1, 4, 64, 0, 32, 0.1), -1),          # no heads
    ((1, 4, 64, 2, 32, float("nan")), -1),  # non-finite scale
    ((1, 4, 64, 2, 24, 0.1), -2),          # unsupported head dim
    ((1, 4, 64, 2, 64, 0.1), -2),
    ((1, 4, 1025, 2, 32, 0.1), -2),        # N above the limit
    ((1, 4, 64, 257, 32, 0.1), -2),        # H above the limit
    ((1, 4, 64, 2, 32, 0.1, 2), -1),       # unknown node
    ((1, 4, 64, 2, 32, 0.1, -1), -1),
])
def test_shape_validation(lib, shape, code):
    assert _fwd(lib, shape) == code
    assert _bwd(lib, shape, 1 << 40) == code


@pytest.mark.parametrize("name", ["Q", "K", "V", "bias", "O", "LSE"])
def test_fwd_null_required_pointer(lib, name):
    assert _fwd(lib, GOOD, **{name: 0}) == -1


@pytest.mark.parametrize("name", ["Q", "K", "V", "bias", "mask", "O", "LSE", "Ores"])
def test_fwd_misaligned_pointer(lib, name):
    assert _fwd(lib, GOOD, **{name: FAKE + 2}) == -2


@pytest.mark.parametrize("name", ["Q", "K", "V", "bias", "O", "LSE", "dO", "dQ", "dK", "dV", "dBias"])
def test_bwd_null_required_pointer(lib, name):
    assert _bwd(lib, GOOD, 1 << 40, **{name: 0}) == -1


def test_bwd_workspace_checks(lib):
    from bwd_tri_attn_gb300.binding import Shape
    need = lib.tri_attn_bwd_workspace_size(Shape(*GOOD))
    assert _bwd(lib, GOOD, 1 << 40, ws=FAKE + 8) == -2  # a misaligned workspace, before any device query
    if not _has_device():
        # the size bound depends on the device's SM count: without a device there is none, and a
        # call with valid arguments is refused on the host (nothing can be launched)
        assert need == 0
        assert _bwd(lib, GOOD, 1 << 40) == -4
        return
    assert need > 0
    assert _bwd(lib, GOOD, need - 1) == -3
    assert _bwd(lib, GOOD, need, ws=0) == -3


def test_workspace_size_depends_on_shape_and_device_only(lib):
    from bwd_tri_attn_gb300.binding import Shape
    a = lib.tri_attn_bwd_workspace_size(Shape(1, 768, 768, 4, 32, 0.1))
    b = lib.tri_attn_bwd_workspace_size(Shape(1, 768, 768, 4, 32, 0.5))
    assert a == b
    assert lib.tri_attn_bwd_workspace_size(Shape(1, 768, 768, 4, 24, 0.1)) == 0
    if _has_device():
        # at least the FP32 correction D [B,S,H,N]
        assert a >= 4 * 768 * 4 * 768
    else:
        assert a == 0


def test_split_query_validation(lib):
    from bwd_tri_attn_gb300.binding import Shape
    nc, k = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.tri_attn_bwd_split(Shape(1, 4, 64, 2, 24, 0.1), 0, ctypes.byref(nc), ctypes.byref(k)) == -2
    assert lib.tri_attn_bwd_split(Shape(*GOOD), 0, None, ctypes.byref(k)) == -1
    assert lib.tri_attn_bwd_split(Shape(*GOOD), 1, ctypes.byref(nc), None) == -1
    # too large for the static array: refused from the shape alone, device or not
    assert lib.tri_attn_bwd_split(Shape(1, 1024, 1024, 4, 32, 0.1), 1, ctypes.byref(nc), ctypes.byref(k)) == -6
    rc = lib.tri_attn_bwd_split(Shape(*GOOD), 0, ctypes.byref(nc), ctypes.byref(k))
    if _has_device():
        assert rc == 0 and nc.value >= 1 and k.value >= 1
    else:
        assert rc == -4


def test_timing_events_validation(lib):
    assert lib.tri_attn_set_timing_events(None, -1) == -1
    assert lib.tri_attn_set_timing_events(None, 0) == 0


def test_workspace_size_same_for_both_nodes(lib):
    from bwd_tri_attn_gb300.binding import Shape
    lib.tri_attn_bwd_workspace_size.restype = ctypes.c_size_t
    a = lib.tri_attn_bwd_workspace_size(Shape(1, 96, 200, 4, 32, 0.17677669, 0))
    b = lib.tri_attn_bwd_workspace_size(Shape(1, 96, 200, 4, 32, 0.17677669, 1))
    assert a == b
    assert (a > 0) == _has_device()


# ---------------------------------------------------------------- triangle multiplication entry points
MUL_GOOD = (1, 64, 16, 0, 0)


def _mul_fwd(lib, shape, **ptrs):
    from bwd_tri_attn_gb300.binding import MulShape
    names = ["Pa", "Ga", "Pb", "Gb", "A", "Bm", "X"]
    args = [ctypes.c_void_p(ptrs.get(n, FAKE)) for n in names]
    return lib.tri_mul_fwd(MulShape(*shape), *args, None)


def _mul_bwd(lib, shape, ws_bytes, **ptrs):
    from bwd_tri_attn_gb300.binding import MulShape
    names = ["Pa", "Ga", "Pb", "Gb", "A", "Bm", "dX", "dPa", "dGa", "dPb", "dGb", "ws"]
    args = [ctypes.c_void_p(ptrs.get(n, FAKE)) for n in names]
    return lib.tri_mul_bwd(MulShape(*shape), *args, ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("shape,code", [
    ((0, 64, 16, 0, 0), -1),      # empty batch
    ((1, 0, 16, 0, 0), -1),       # no residues
    ((1, 64, 0, 0, 0), -1),       # no channels
    ((1, 64, 16, 2, 0), -1),      # unknown direction
    ((1, 64, 16, -1, 0), -1),
    ((1, 64, 16, 0, 2), -1),      # unknown layout
    ((1, 64, 16, 0, -1), -1),
    ((1, 8, 16, 0, 0), -2),       # N below 16
    ((1, 68, 16, 0, 1), -2),      # N not a multiple of 8
    ((1, 4104, 16, 0, 0), -2),    # N above TRI_MUL_MAX_N
    ((1, 64, 12, 0, 1), -2),      # C not a multiple of 8
    ((1, 64, 1032, 0, 0), -2),    # C above TRI_MUL_MAX_C
    ((65, 64, 1024, 0, 1), -2),   # B * C above the grid limit
])
def test_mul_shape_validation(lib, shape, code):
    assert _mul_fwd(lib, shape) == code
    assert _mul_bwd(lib, shape, 1 << 40) == code


@pytest.mark.parametrize("name", ["Pa", "Ga", "Pb", "Gb", "A", "Bm", "X"])
def test_mul_fwd_pointer_checks(lib, name):
    assert _mul_fwd(lib, MUL_GOOD, **{name: 0}) == -1
    assert _mul_fwd(lib, MUL_GOOD, **{name: FAKE + 2}) == -2


@pytest.mark.parametrize("name", ["Pa", "Ga", "Pb", "Gb", "A", "Bm", "dX", "dPa", "dGa", "dPb", "dGb"])
def test_mul_bwd_pointer_checks(lib, name):
    assert _mul_bwd(lib, MUL_GOOD, 1 << 40, **{name: 0}) == -1
    assert _mul_bwd(lib, MUL_GOOD, 1 << 40, **{name: FAKE + 2}) == -2


def test_mul_workspace_checks(lib):
    from bwd_tri_attn_gb300.binding import MulShape
    need = lib.tri_mul_bwd_workspace_size(MulShape(*MUL_GOOD))
    assert need == 2 * 4 * 1 * 16 * 64 * 64  # two FP32 [B, C, N, N] stacks, known without a device
    assert lib.tri_mul_bwd_workspace_size(MulShape(1, 68, 16, 0, 0)) == 0
    assert lib.tri_mul_bwd_workspace_size(MulShape(1, 64, 16, 0, 1)) == 0  # channel-major: none
    assert _mul_bwd(lib, MUL_GOOD, need - 1) == -3
    assert _mul_bwd(lib, MUL_GOOD, need, ws=0) == -3
    assert _mul_bwd(lib, MUL_GOOD, need, ws=FAKE + 8) == -2


# ---------------------------------------------------------------- triangle-attention block entry points
MOD_GOOD = (1, 64, 128, 4, 32, 0, 1e-5)


def _mod_saved(lib, shape):
    from bwd_tri_attn_gb300.binding import ModuleShape
    return lib.tri_module_saved_size(ModuleShape(*shape))


def _mod_fwd(lib, shape, saved_bytes, **ptrs):
    from bwd_tri_attn_gb300.binding import ModuleShape
    names = ["z", "gamma", "beta", "W", "wb", "Wo", "mask", "out", "saved"]
    args = [ctypes.c_void_p(ptrs.get(n, FAKE)) for n in names]
    return lib.tri_module_fwd(ModuleShape(*shape), *args[:9], ctypes.c_size_t(saved_bytes), None)


def _mod_bwd(lib, shape, saved_bytes, ws_bytes, **ptrs):
    from bwd_tri_attn_gb300.binding import ModuleShape
    pre = [ctypes.c_void_p(ptrs.get(n, FAKE)) for n in ["z", "gamma", "beta", "W", "wb", "Wo", "mask", "saved"]]
    post = [ctypes.c_void_p(ptrs.get(n, FAKE)) for n in ["dout", "dz", "dgamma", "dbeta", "dW", "dwb", "dWo", "ws"]]
    return lib.tri_module_bwd(ModuleShape(*shape), *pre, ctypes.c_size_t(saved_bytes), *post,
                              ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("shape,code", [
    ((0, 64, 128, 4, 32, 0, 1e-5), -1),     # empty batch
    ((1, 64, 128, 0, 32, 0, 1e-5), -1),     # no heads
    ((1, 64, 128, 4, 32, 2, 1e-5), -1),     # unknown node
    ((1, 64, 128, 4, 32, 0, 0.0), -1),      # eps must be positive
    ((1, 64, 128, 4, 32, 0, float("nan")), -1),
    ((1, 64, 96, 4, 32, 0, 1e-5), -2),      # c not 64, 128 or 256
    ((1, 64, 128, 4, 24, 0, 1e-5), -2),     # d not 16 or 32
    ((1, 64, 128, 2, 16, 0, 1e-5), -2),     # H d not a multiple of 64
    ((1, 64, 128, 16, 32, 0, 1e-5), -2),    # more than 8 heads
    ((1, 8, 128, 4, 32, 0, 1e-5), -2),      # N below 16
    ((1, 1032, 128, 4, 32, 0, 1e-5), -2),   # N above the attention's limit
    ((128, 1024, 64, 4, 16, 0, 1e-5), -2),  # B N above the grid limit
])
def test_module_shape_validation(lib, shape, code):
    assert _mod_saved(lib, shape) == 0
    from bwd_tri_attn_gb300.binding import ModuleShape
    assert lib.tri_module_bwd_workspace_size(ModuleShape(*shape)) == 0
    assert _mod_fwd(lib, shape, 1 << 40) == code
    assert _mod_bwd(lib, shape, 1 << 40, 1 << 40) == code


@pytest.mark.parametrize("name", ["z", "gamma", "beta", "W", "wb", "Wo", "out", "saved"])
def test_module_fwd_pointer_checks(lib, name):
    assert _mod_fwd(lib, MOD_GOOD, 1 << 40, **{name: 0}) == -1
    assert _mod_fwd(lib, MOD_GOOD, 1 << 40, **{name: FAKE + 2}) == -2


@pytest.mark.parametrize("name", ["z", "gamma", "beta", "W", "wb", "Wo", "saved", "dout", "dz", "dgamma", "dbeta",
                                  "dW", "dwb", "dWo"])
def test_module_bwd_pointer_checks(lib, name):
    assert _mod_bwd(lib, MOD_GOOD, 1 << 40, 1 << 40, **{name: 0}) == -1
    assert _mod_bwd(lib, MOD_GOOD, 1 << 40, 1 << 40, **{name: FAKE + 2}) == -2


def test_module_saved_and_workspace_checks(lib):
    saved = _mod_saved(lib, MOD_GOOD)
    # at least zt, q, k, v, gl, O, Ores and go (BF16) plus the statistics, bias and log-sum-exp
    M, hd, c = 64 * 64, 128, 128
    assert saved >= 2 * M * c + 7 * 2 * M * hd + 2 * 4 * M + 2 * 4 * 64 * 64 + 4 * 64 * 4 * 64
    assert _mod_saved(lib, (1, 64, 128, 4, 32, 1, 1e-5)) == saved  # the node changes no size
    assert _mod_fwd(lib, MOD_GOOD, saved - 1) == -3
    assert _mod_bwd(lib, MOD_GOOD, saved - 1, 1 << 40) == -3
    assert _mod_fwd(lib, MOD_GOOD, saved, mask=FAKE + 4) == -2  # the optional mask is still checked
    assert _mod_bwd(lib, MOD_GOOD, saved, 1 << 40, ws=0) == -3
    if _has_device():
        from bwd_tri_attn_gb300.binding import ModuleShape
        need = lib.tri_module_bwd_workspace_size(ModuleShape(*MOD_GOOD))
        assert need > 0
        assert _mod_bwd(lib, MOD_GOOD, saved, need - 1) == -3


# ---------------------------------------------------------------- binding argument checks
# The C ABI takes bare pointers; the Python binding checks what a pointer cannot carry (dtype,
# contiguity, element count, device) before anything reaches the library.

def _attn_tensors(dtype_over=None, drop=None):
    B, S, N, H, d = 1, 4, 24, 2, 16
    pair = lambda: torch.zeros((B, S, N, H, d), dtype=torch.bfloat16)  # noqa: E731
    t = {"Q": pair(), "K": pair(), "V": pair(), "bias": torch.zeros((B, H, N, N), dtype=torch.bfloat16),
         "mask": None, "O": pair(), "LSE": torch.zeros((B, S, H, N)), "Ores": pair()}
    if dtype_over:
        t[dtype_over[0]] = t[dtype_over[0]].to(dtype_over[1])
    return t


def test_binding_rejects_wrong_tensors_before_the_call():
    import torch
    from bwd_tri_attn_gb300 import binding as tb
    shape = tb.Shape(1, 4, 24, 2, 16, 0.25, 0)
    args = lambda t: (t["Q"], t["K"], t["V"], t["bias"], t["mask"], t["O"], t["LSE"], t["Ores"])  # noqa: E731
    with pytest.raises(TypeError, match="K must be torch.bfloat16"):
        tb.tri_attn_fwd(shape, *args(_attn_tensors(("K", torch.float16))))
    with pytest.raises(TypeError, match="LSE must be torch.float32"):
        tb.tri_attn_fwd(shape, *args(_attn_tensors(("LSE", torch.bfloat16))))
    t = _attn_tensors()
    t["V"] = torch.zeros((1, 4, 2, 24, 16), dtype=torch.bfloat16).transpose(2, 3)  # right shape, strided
    with pytest.raises(ValueError, match="V must be contiguous"):
        tb.tri_attn_fwd(shape, *args(t))
    t = _attn_tensors()
    t["bias"] = torch.zeros((1, 2, 24, 23), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="bias has 1104 elements, the shape needs 1152"):
        tb.tri_attn_fwd(shape, *args(t))
    t = _attn_tensors()
    t["Q"] = None
    with pytest.raises(ValueError, match="Q is required"):
        tb.tri_attn_fwd(shape, *args(t))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):  # everything right but the device
        tb.tri_attn_fwd(shape, *args(_attn_tensors()))


def test_binding_checks_module_and_multiplication_arguments():
    import torch
    from bwd_tri_attn_gb300 import binding as tb
    ms = tb.ModuleShape(1, 16, 64, 2, 32, 0, 1e-5)
    z = torch.zeros((1, 16, 16, 64), dtype=torch.bfloat16)
    gamma, beta = torch.ones(64), torch.zeros(64)
    W, wb, Wo = (torch.zeros(s, dtype=torch.bfloat16) for s in ((256, 64), (2, 64), (64, 64)))
    with pytest.raises(TypeError, match="gamma must be torch.float32"):
        tb.tri_module_fwd(ms, z, gamma.bfloat16(), beta, W, wb, Wo, None, torch.empty_like(z), None)
    with pytest.raises(ValueError, match="W has 8192 elements, the shape needs 16384"):
        tb.tri_module_fwd(ms, z, gamma, beta, W[:128], wb, Wo, None, torch.empty_like(z), None)
    mu = tb.MulShape(1, 16, 32, 0, tb.LAYOUT_PAIR)
    P = [torch.zeros((1, 16, 16, 32), dtype=torch.bfloat16) for _ in range(7)]
    P[5] = P[5][:, :8]
    with pytest.raises(ValueError, match="Bm must be contiguous|Bm has"):
        tb.tri_mul_fwd(mu, *P)


def test_binding_module_backward_reaches_the_device_check():
    # every argument of the block's backward well-formed on the host: the only complaint left is the
    # device, so the argument list itself is assembled completely
    import torch
    from bwd_tri_attn_gb300 import binding as tb
    ms = tb.ModuleShape(1, 16, 64, 2, 32, 0, 1e-5)
    z = torch.zeros((1, 16, 16, 64), dtype=torch.bfloat16)
    gamma, beta = torch.ones(64), torch.zeros(64)
    W, wb, Wo = (torch.zeros(s, dtype=torch.bfloat16) for s in ((256, 64), (2, 64), (64, 64)))
    saved, ws = torch.zeros(64, dtype=torch.uint8), torch.zeros(64, dtype=torch.uint8)
    grads = [torch.zeros(s) for s in ((64,), (64,), (256, 64), (2, 64), (64, 64))]
    with pytest.raises(ValueError, match="z must be a CUDA tensor"):
        tb.tri_module_bwd(ms, z, gamma, beta, W, wb, Wo, None, saved, z, torch.empty_like(z), *grads, ws)
    with pytest.raises(TypeError, match="dW must be torch.float32"):
        tb.tri_module_bwd(ms, z, gamma, beta, W, wb, Wo, None, saved, z, torch.empty_like(z), grads[0], grads[1],
                          grads[2].bfloat16(), grads[3], grads[4], ws)
