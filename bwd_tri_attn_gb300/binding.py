"""Thin ctypes binding of the C ABI in ``include/tri_attn.h``, ``include/tri_mul.h`` and
``include/tri_module.h``.

Argument marshalling only: PyTorch tensors supply device pointers and the
current CUDA stream; every step of the computation runs in the library's
kernels. There is no CPU fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

TRI_ATTN_OK = 0
_lock = threading.Lock()
_lib = None


NODE_STARTING, NODE_ENDING = 0, 1  # tri_attn_shape.node


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("S", ctypes.c_int), ("N", ctypes.c_int), ("H", ctypes.c_int),
                ("d", ctypes.c_int), ("scale", ctypes.c_float), ("node", ctypes.c_int)]

    def __repr__(self):
        return (f"Shape(B={self.B}, S={self.S}, N={self.N}, H={self.H}, d={self.d}, scale={self.scale}, "
                f"node={self.node})")


class TriAttnError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")
        self.code = code


_VP = ctypes.c_void_p
EXPORTS = ("tri_attn_strerror", "tri_attn_fwd", "tri_attn_bwd_workspace_size", "tri_attn_bwd_split", "tri_attn_bwd",
           "tri_attn_device_status", "tri_attn_set_timing_events", "tri_attn_bwd_static", "tri_mul_fwd",
           "tri_mul_bwd_workspace_size", "tri_mul_bwd", "tri_module_saved_size", "tri_module_bwd_workspace_size",
           "tri_module_fwd", "tri_module_bwd")


LAYOUT_PAIR, LAYOUT_CHANNEL_MAJOR = 0, 1  # tri_mul_shape.layout


class MulShape(ctypes.Structure):
    """tri_mul_shape: batch, residues, channels, direction (0 outgoing, 1 incoming), layout of the
    projections and their gradients (LAYOUT_PAIR [B,N,N,C] or LAYOUT_CHANNEL_MAJOR [B,C,N,N])."""
    _fields_ = [("B", ctypes.c_int), ("N", ctypes.c_int), ("C", ctypes.c_int), ("incoming", ctypes.c_int),
                ("layout", ctypes.c_int)]

    def __repr__(self):
        return (f"MulShape(B={self.B}, N={self.N}, C={self.C}, incoming={self.incoming}, "
                f"layout={self.layout})")


class ModuleShape(ctypes.Structure):
    """tri_module_shape: batch, residues, pair channels, heads, head dimension, node, LayerNorm eps."""
    _fields_ = [("B", ctypes.c_int), ("N", ctypes.c_int), ("c", ctypes.c_int), ("H", ctypes.c_int),
                ("d", ctypes.c_int), ("node", ctypes.c_int), ("eps", ctypes.c_float)]

    def __repr__(self):
        return (f"ModuleShape(B={self.B}, N={self.N}, c={self.c}, H={self.H}, d={self.d}, node={self.node}, "
                f"eps={self.eps})")


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Loads ``libtriattn.so`` (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first (__graft_entry__.build())")
        lib = ctypes.CDLL(path)
        lib.tri_attn_strerror.argtypes = [ctypes.c_int]
        lib.tri_attn_strerror.restype = ctypes.c_char_p
        lib.tri_attn_fwd.argtypes = [Shape] + [_VP] * 9
        lib.tri_attn_fwd.restype = ctypes.c_int
        lib.tri_attn_bwd_workspace_size.argtypes = [Shape]
        lib.tri_attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.tri_attn_bwd_split.argtypes = [Shape, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_int)]
        lib.tri_attn_bwd_split.restype = ctypes.c_int
        lib.tri_attn_bwd.argtypes = [Shape] + [_VP] * 14 + [ctypes.c_size_t, _VP]
        lib.tri_attn_bwd.restype = ctypes.c_int
        lib.tri_attn_device_status.argtypes = [_VP]
        lib.tri_attn_device_status.restype = ctypes.c_int
        lib.tri_attn_bwd_static.argtypes = [Shape] + [_VP] * 14
        lib.tri_attn_bwd_static.restype = ctypes.c_int
        lib.tri_attn_set_timing_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
        lib.tri_attn_set_timing_events.restype = ctypes.c_int
        lib.tri_mul_fwd.argtypes = [MulShape] + [_VP] * 8
        lib.tri_mul_fwd.restype = ctypes.c_int
        lib.tri_mul_bwd_workspace_size.argtypes = [MulShape]
        lib.tri_mul_bwd_workspace_size.restype = ctypes.c_size_t
        lib.tri_mul_bwd.argtypes = [MulShape] + [_VP] * 12 + [ctypes.c_size_t, _VP]
        lib.tri_mul_bwd.restype = ctypes.c_int
        lib.tri_module_saved_size.argtypes = [ModuleShape]
        lib.tri_module_saved_size.restype = ctypes.c_size_t
        lib.tri_module_bwd_workspace_size.argtypes = [ModuleShape]
        lib.tri_module_bwd_workspace_size.restype = ctypes.c_size_t
        lib.tri_module_fwd.argtypes = [ModuleShape] + [_VP] * 9 + [ctypes.c_size_t, _VP]
        lib.tri_module_fwd.restype = ctypes.c_int
        lib.tri_module_bwd.argtypes = [ModuleShape] + [_VP] * 8 + [ctypes.c_size_t] + [_VP] * 8 + [ctypes.c_size_t, _VP]
        lib.tri_module_bwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load().tri_attn_strerror(int(code)).decode()


def shape_of(Q: torch.Tensor, scale: float | None = None, node: int = NODE_STARTING) -> Shape:
    """Shape of the attention on the pair tensor Q: [B, S, N, H, d] for the starting node (slices
    along pair axis 1), [B, N, S, H, d] for the ending node (slices along pair axis 2)."""
    B, P1, P2, H, d = (int(x) for x in Q.shape)
    S, N = (P1, P2) if node == NODE_STARTING else (P2, P1)
    return Shape(B, S, N, H, d, float(1.0 / math.sqrt(d) if scale is None else scale), int(node))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


_BF16, _F32 = torch.bfloat16, torch.float32


def _arg(t, name, dtype, numel, nullable=False):
    """Checks tensor argument `name` for what the C ABI cannot check on a bare pointer: dtype,
    contiguity and the element count the shape implies (None: any). Returns it for _ptrs, which
    checks the devices once every argument has passed these checks."""
    if t is None:
        if nullable:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, the shape needs {numel}")
    return (name, t)


def _ptrs(*checked):
    """Device pointers of arguments that passed _arg: each a CUDA tensor on the current device (a
    wrong tensor raises here instead of being read or written out of bounds)."""
    out = []
    for c in checked:
        if c is None:
            out.append(None)
            continue
        name, t = c
        if not t.is_cuda or t.device.index != torch.cuda.current_device():
            raise ValueError(f"{name} must be a CUDA tensor on the current device, got {t.device}")
        out.append(ctypes.c_void_p(t.data_ptr()))
    return out


def _attn_counts(shape):
    pair = shape.B * shape.S * shape.N * shape.H * shape.d
    return pair, shape.B * shape.H * shape.N * shape.N, shape.B * shape.S * shape.N, shape.B * shape.S * shape.H * shape.N


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn, rc):
    if rc != TRI_ATTN_OK:
        raise TriAttnError(fn, rc)


def tri_attn_fwd(shape: Shape, Q, K, V, bias, mask, O, LSE, Ores, stream=None):
    pair, nb, nm, nl = _attn_counts(shape)
    ptrs = _ptrs(_arg(Q, "Q", _BF16, pair), _arg(K, "K", _BF16, pair), _arg(V, "V", _BF16, pair),
                 _arg(bias, "bias", _BF16, nb), _arg(mask, "mask", _BF16, nm, True), _arg(O, "O", _BF16, pair),
                 _arg(LSE, "LSE", _F32, nl), _arg(Ores, "Ores", _BF16, pair, True))
    rc = load().tri_attn_fwd(shape, *ptrs, _stream(stream))
    _check("tri_attn_fwd", rc)


def tri_attn_bwd_workspace_size(shape: Shape) -> int:
    return int(load().tri_attn_bwd_workspace_size(shape))


def tri_attn_bwd_split(shape: Shape, static_entry: bool = False) -> tuple[int, int]:
    """(clusters, dBias partial slots per head) of the backward's work split on the current device."""
    nc, slots = ctypes.c_int(0), ctypes.c_int(0)
    rc = load().tri_attn_bwd_split(shape, int(bool(static_entry)), ctypes.byref(nc), ctypes.byref(slots))
    _check("tri_attn_bwd_split", rc)
    return nc.value, slots.value


def _attn_bwd_args(shape, Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias):
    pair, nb, nm, nl = _attn_counts(shape)
    return [_arg(Q, "Q", _BF16, pair), _arg(K, "K", _BF16, pair), _arg(V, "V", _BF16, pair),
            _arg(bias, "bias", _BF16, nb), _arg(mask, "mask", _BF16, nm, True), _arg(O, "O", _BF16, pair),
            _arg(Ores, "Ores", _BF16, pair, True), _arg(LSE, "LSE", _F32, nl), _arg(dO, "dO", _BF16, pair),
            _arg(dQ, "dQ", _BF16, pair), _arg(dK, "dK", _BF16, pair), _arg(dV, "dV", _BF16, pair),
            _arg(dBias, "dBias", _BF16, nb)]


def tri_attn_bwd(shape: Shape, Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias, workspace,
                 stream=None):
    ptrs = _ptrs(*_attn_bwd_args(shape, Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias),
                 _arg(workspace, "workspace", None, None, True))
    rc = load().tri_attn_bwd(shape, *ptrs, _nbytes(workspace), _stream(stream))
    _check("tri_attn_bwd", rc)


def tri_attn_bwd_static(shape: Shape, Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias, stream=None):
    """Backward pass with the library's static scratch array (no workspace argument)."""
    ptrs = _ptrs(*_attn_bwd_args(shape, Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias))
    rc = load().tri_attn_bwd_static(shape, *ptrs, _stream(stream))
    _check("tri_attn_bwd_static", rc)


def tri_mul_fwd(shape: MulShape, Pa, Ga, Pb, Gb, A, Bm, X, stream=None):
    n = shape.B * shape.N * shape.N * shape.C
    ptrs = _ptrs(*[_arg(t, k, _BF16, n) for t, k in ((Pa, "Pa"), (Ga, "Ga"), (Pb, "Pb"), (Gb, "Gb"), (A, "A"),
                                                     (Bm, "Bm"), (X, "X"))])
    rc = load().tri_mul_fwd(shape, *ptrs, _stream(stream))
    _check("tri_mul_fwd", rc)


def tri_mul_bwd_workspace_size(shape: MulShape) -> int:
    return int(load().tri_mul_bwd_workspace_size(shape))


def tri_mul_bwd(shape: MulShape, Pa, Ga, Pb, Gb, A, Bm, dX, dPa, dGa, dPb, dGb, workspace, stream=None):
    n = shape.B * shape.N * shape.N * shape.C
    ptrs = _ptrs(*[_arg(t, k, _BF16, n) for t, k in ((Pa, "Pa"), (Ga, "Ga"), (Pb, "Pb"), (Gb, "Gb"), (A, "A"),
                                                     (Bm, "Bm"), (dX, "dX"), (dPa, "dPa"), (dGa, "dGa"),
                                                     (dPb, "dPb"), (dGb, "dGb"))],
                 _arg(workspace, "workspace", None, None, True))
    rc = load().tri_mul_bwd(shape, *ptrs, _nbytes(workspace), _stream(stream))
    _check("tri_mul_bwd", rc)


def tri_module_saved_size(shape: ModuleShape) -> int:
    return int(load().tri_module_saved_size(shape))


def tri_module_bwd_workspace_size(shape: ModuleShape) -> int:
    return int(load().tri_module_bwd_workspace_size(shape))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _module_args(shape, z, gamma, beta, W, wb, Wo, mask):
    B, N, c, hd = shape.B, shape.N, shape.c, shape.H * shape.d
    return [_arg(z, "z", _BF16, B * N * N * c), _arg(gamma, "gamma", _F32, c), _arg(beta, "beta", _F32, c),
            _arg(W, "W", _BF16, 4 * hd * c), _arg(wb, "wb", _BF16, shape.H * c), _arg(Wo, "Wo", _BF16, c * hd),
            _arg(mask, "mask", _BF16, B * N * N, True)]


def tri_module_fwd(shape: ModuleShape, z, gamma, beta, W, wb, Wo, mask, out, saved, stream=None):
    n = shape.B * shape.N * shape.N * shape.c
    ptrs = _ptrs(*_module_args(shape, z, gamma, beta, W, wb, Wo, mask), _arg(out, "out", _BF16, n),
                 _arg(saved, "saved", None, None, True))
    rc = load().tri_module_fwd(shape, *ptrs, _nbytes(saved), _stream(stream))
    _check("tri_module_fwd", rc)


def tri_module_bwd(shape: ModuleShape, z, gamma, beta, W, wb, Wo, mask, saved, dout, dz, dgamma, dbeta, dW, dwb,
                   dWo, workspace, stream=None):
    n, c, hd = shape.B * shape.N * shape.N * shape.c, shape.c, shape.H * shape.d
    p = _ptrs(*_module_args(shape, z, gamma, beta, W, wb, Wo, mask), _arg(saved, "saved", None, None, True),
              _arg(dout, "dout", _BF16, n), _arg(dz, "dz", _BF16, n), _arg(dgamma, "dgamma", _F32, c),
              _arg(dbeta, "dbeta", _F32, c), _arg(dW, "dW", _F32, 4 * hd * c), _arg(dwb, "dwb", _F32, shape.H * c),
              _arg(dWo, "dWo", _F32, c * hd), _arg(workspace, "workspace", None, None, True))
    # (z .. mask, saved | dout .. dWo, workspace)
    rc = load().tri_module_bwd(shape, *p[:8], _nbytes(saved), *p[8:16], _nbytes(workspace), _stream(stream))
    _check("tri_module_bwd", rc)


def tri_attn_device_status(stream=None) -> int:
    return int(load().tri_attn_device_status(_stream(stream)))


_event_array = None  # keeps the pointer array alive while instrumentation is on


def tri_attn_set_timing_events(events) -> None:
    """Per-kernel timing: ``events`` is a list of recorded torch.cuda.Event (or None to switch off)."""
    global _event_array
    if not events:
        _event_array = None
        _check("tri_attn_set_timing_events", load().tri_attn_set_timing_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _event_array = arr
    _check("tri_attn_set_timing_events", load().tri_attn_set_timing_events(arr, len(events)))


# ----------------------------------------------------------------------------
# Allocating conveniences (outputs are fresh torch tensors on Q's device).
# ----------------------------------------------------------------------------

def forward(Q, K, V, bias, mask=None, scale=None, residual=True, stream=None, node=NODE_STARTING):
    """Returns (O, LSE, Ores); Ores is None when ``residual`` is False. O and Ores have Q's
    layout; LSE is [B, S, H, N] in terms of the attention's slices and positions."""
    shape = shape_of(Q, scale, node)
    B, S, N, H = shape.B, shape.S, shape.N, shape.H
    O = torch.empty_like(Q)
    LSE = torch.empty((B, S, H, N), dtype=torch.float32, device=Q.device)
    Ores = torch.empty_like(Q) if residual else None
    tri_attn_fwd(shape, Q, K, V, bias, mask, O, LSE, Ores, stream)
    return O, LSE, Ores


def workspace_for(shape: Shape, device) -> torch.Tensor:
    n = tri_attn_bwd_workspace_size(shape)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def backward(Q, K, V, bias, mask, O, Ores, LSE, dO, scale=None, workspace=None, stream=None,
             node=NODE_STARTING):
    """Returns (dQ, dK, dV, dBias)."""
    shape = shape_of(Q, scale, node)
    if workspace is None:
        workspace = workspace_for(shape, Q.device)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    dBias = torch.empty_like(bias)
    tri_attn_bwd(shape, Q, K, V, bias, mask, O, Ores, LSE, dO, dQ, dK, dV, dBias, workspace, stream)
    return dQ, dK, dV, dBias


def mul_shape_of(Pa: torch.Tensor, incoming: bool = False, layout: int = LAYOUT_PAIR) -> MulShape:
    """Shape of the triangle multiplicative update on projections [B, N, N, C] (pair layout) or
    [B, C, N, N] (channel-major)."""
    if layout == LAYOUT_PAIR:
        B, N, N2, C = (int(x) for x in Pa.shape)
    else:
        B, C, N, N2 = (int(x) for x in Pa.shape)
    if N2 != N:
        raise ValueError(f"projection must be square in its two position axes, got {tuple(Pa.shape)}")
    return MulShape(B, N, C, int(bool(incoming)), int(layout))


def mul_forward(Pa, Ga, Pb, Gb, incoming=False, layout=LAYOUT_PAIR, stream=None):
    """Returns (X, A, Bm): X [B, C, N, N] channel-major, and the gated operands A, Bm
    [B, C, N, N] that mul_backward reads."""
    shape = mul_shape_of(Pa, incoming, layout)
    B, N, C = shape.B, shape.N, shape.C
    A, Bm, X = (torch.empty((B, C, N, N), dtype=torch.bfloat16, device=Pa.device) for _ in range(3))
    tri_mul_fwd(shape, Pa, Ga, Pb, Gb, A, Bm, X, stream)
    return X, A, Bm


def mul_backward(Pa, Ga, Pb, Gb, A, Bm, dX, incoming=False, layout=LAYOUT_PAIR, workspace=None, stream=None):
    """Returns (dPa, dGa, dPb, dGb) in the projections' layout; dX is channel-major."""
    shape = mul_shape_of(Pa, incoming, layout)
    if workspace is None:
        workspace = torch.empty(max(tri_mul_bwd_workspace_size(shape), 16), dtype=torch.uint8, device=Pa.device)
    outs = [torch.empty_like(Pa) for _ in range(4)]
    tri_mul_bwd(shape, Pa, Ga, Pb, Gb, A, Bm, dX, *outs, workspace, stream)
    return tuple(outs)


def module_shape_of(z: torch.Tensor, H: int, d: int, node: int = NODE_STARTING, eps: float = 1e-5) -> ModuleShape:
    """Shape of the triangle-attention block on the pair representation z [B, N, N, c]."""
    B, N, N2, c = (int(x) for x in z.shape)
    if N2 != N:
        raise ValueError(f"pair representation must be square, got {tuple(z.shape)}")
    return ModuleShape(B, N, c, int(H), int(d), int(node), float(eps))


def module_forward(z, gamma, beta, W, wb, Wo, mask, H, d, node=NODE_STARTING, eps=1e-5, stream=None):
    """Returns (out, saved): out [B, N, N, c] and the activations module_backward reads."""
    shape = module_shape_of(z, H, d, node, eps)
    saved = torch.empty(max(tri_module_saved_size(shape), 16), dtype=torch.uint8, device=z.device)
    out = torch.empty_like(z)
    tri_module_fwd(shape, z, gamma, beta, W, wb, Wo, mask, out, saved, stream)
    return out, saved


def module_backward(z, gamma, beta, W, wb, Wo, mask, saved, dout, H, d, node=NODE_STARTING, eps=1e-5,
                    workspace=None, stream=None):
    """Returns (dz, dgamma, dbeta, dW, dwb, dWo); the weight gradients are FP32."""
    shape = module_shape_of(z, H, d, node, eps)
    if workspace is None:
        workspace = torch.empty(max(tri_module_bwd_workspace_size(shape), 16), dtype=torch.uint8, device=z.device)
    dz = torch.empty_like(z)
    f32 = dict(dtype=torch.float32, device=z.device)
    dgamma, dbeta = torch.empty(gamma.shape, **f32), torch.empty(beta.shape, **f32)
    dW, dwb, dWo = torch.empty(W.shape, **f32), torch.empty(wb.shape, **f32), torch.empty(Wo.shape, **f32)
    tri_module_bwd(shape, z, gamma, beta, W, wb, Wo, mask, saved, dout, dz, dgamma, dbeta, dW, dwb, dWo, workspace,
                   stream)
    return dz, dgamma, dbeta, dW, dwb, dWo
