"""FP64 CPU oracle for triangle attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The CUDA library never links, loads or
calls it, and the two share no code.

The arithmetic lives in ``tri_attn_oracle.c`` (plain C, double precision,
OpenMP over independent (batch, slice, head) items); this module only builds
that file with gcc and marshals numpy float64 arrays through ctypes.

Definition followed (TurboPairFormer, arXiv 2610.05854v1, Abstract): each
row-slice of the pair tensor runs multi-head attention with a pair bias shared
by all slices, so the bias gradient is the slice-sum of the per-slice score
gradients.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tri_attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DP = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compiles the oracle into ``oracle/liboracle.so`` (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            shape = [ctypes.c_int] * 5 + [ctypes.c_double]
            lib.oracle_tri_attn_fwd.argtypes = shape + [_DP] * 7 + [ctypes.c_int]
            lib.oracle_tri_attn_fwd.restype = ctypes.c_int
            lib.oracle_tri_attn_bwd.argtypes = shape + [_DP] * 11 + [ctypes.c_int]
            lib.oracle_tri_attn_bwd.restype = ctypes.c_int
            lib.oracle_tri_attn_slice.argtypes = shape + [ctypes.c_int] * 3 + [_DP] * 8
            lib.oracle_tri_attn_slice.restype = ctypes.c_int
            lib.oracle_tri_attn_dbias_rows.argtypes = shape + [_DP] * 6 + [ctypes.POINTER(ctypes.c_int), ctypes.c_int, _DP, ctypes.c_int]
            lib.oracle_tri_attn_dbias_rows.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (any dtype) -> exact float64 copy
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_DP)


def _dims(Q):
    B, S, N, H, d = Q.shape
    return int(B), int(S), int(N), int(H), int(d)


def num_threads(nthreads: int = 0) -> int:
    """Threads the oracle's parallel regions use for a request (0 = OpenMP default)."""
    return int(_load().oracle_num_threads(int(nthreads)))


def fwd(Q, K, V, bias, mask=None, scale=None, nthreads: int = 0):
    """Returns (O [B,S,N,H,d], LSE [B,S,H,N]) in float64.

    Q, K, V: [B,S,N,H,d]; bias: [B,H,N,N]; mask: [B,S,N] additive or None.
    scale defaults to 1/sqrt(d).
    """
    Q, K, V, bias, mask = (_f64(t) for t in (Q, K, V, bias, mask))
    B, S, N, H, d = _dims(Q)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    O = np.zeros((B, S, N, H, d))
    LSE = np.zeros((B, S, H, N))
    rc = _load().oracle_tri_attn_fwd(B, S, N, H, d, scale, _ptr(Q), _ptr(K), _ptr(V),
                                     _ptr(bias), _ptr(mask), _ptr(O), _ptr(LSE), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_tri_attn_fwd failed: {rc}")
    return O, LSE


def bwd(Q, K, V, bias, mask, dO, scale=None, nthreads: int = 0):
    """Returns dict with dQ, dK, dV [B,S,N,H,d], dBias [B,H,N,N], D [B,S,H,N] (float64)."""
    Q, K, V, bias, mask, dO = (_f64(t) for t in (Q, K, V, bias, mask, dO))
    B, S, N, H, d = _dims(Q)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = {k: np.zeros((B, S, N, H, d)) for k in ("dQ", "dK", "dV")}
    out["dBias"] = np.zeros((B, H, N, N))
    out["D"] = np.zeros((B, S, H, N))
    rc = _load().oracle_tri_attn_bwd(B, S, N, H, d, scale, _ptr(Q), _ptr(K), _ptr(V),
                                     _ptr(bias), _ptr(mask), _ptr(dO), _ptr(out["dQ"]),
                                     _ptr(out["dK"]), _ptr(out["dV"]), _ptr(out["dBias"]),
                                     _ptr(out["D"]), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_tri_attn_bwd failed: {rc}")
    return out


def slice_matrices(Q, K, V, bias, mask, dO, b, i, h, scale=None):
    """Materialised P and dS [N,N] of one (b,i,h) slice (dS is None when dO is None)."""
    Q, K, V, bias, mask, dO = (_f64(t) for t in (Q, K, V, bias, mask, dO))
    B, S, N, H, d = _dims(Q)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    P = np.zeros((N, N))
    dS = np.zeros((N, N)) if dO is not None else None
    rc = _load().oracle_tri_attn_slice(B, S, N, H, d, scale, int(b), int(i), int(h), _ptr(Q),
                                       _ptr(K), _ptr(V), _ptr(bias), _ptr(mask), _ptr(dO),
                                       _ptr(P), _ptr(dS))
    if rc != 0:
        raise RuntimeError(f"oracle_tri_attn_slice failed: {rc}")
    return P, dS


def dbias_rows(Q, K, V, bias, mask, dO, rows, scale=None, nthreads: int = 0):
    """dBias[b,h,j,:] for each (b,h,j) in ``rows``, summed over all slices: array [len(rows), N]."""
    Q, K, V, bias, mask, dO = (_f64(t) for t in (Q, K, V, bias, mask, dO))
    B, S, N, H, d = _dims(Q)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    out = np.zeros((r.shape[0], N))
    rc = _load().oracle_tri_attn_dbias_rows(B, S, N, H, d, scale, _ptr(Q), _ptr(K), _ptr(V), _ptr(bias),
                                            _ptr(mask), _ptr(dO),
                                            r.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), r.shape[0],
                                            _ptr(out), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_tri_attn_dbias_rows failed: {rc}")
    return out
