"""fp64 oracle for the CP state-correction pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library's CUDA path never calls it and shares
no code with it.  The arithmetic lives in ``qla_oracle.c``; this module only
marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIBS = {}


def _lib(variant: str = ""):
    if variant not in _LIBS:
        path = _build.library_path(variant)
        if not os.path.exists(path):
            if variant:
                raise FileNotFoundError(path)
            _build.build()
        lib = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        ci = ctypes.c_int
        lib.qla_oracle_cp_correct.argtypes = [f32p, f32p, f32p, f64p, f64p, ctypes.c_int64,
                                              ci, ci, ci, ci, ci, ci]
        lib.qla_oracle_cp_correct.restype = ci
        _LIBS[variant] = lib
    return _LIBS[variant]


def _f32(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def cp_correct(H, M, h_init, layout="kv", direction="fwd", want_out=True, want_final=False,
               nthreads=0, variant="", return_threads=False):
    """Exclusive corrected states (and optionally the final state) in fp64.

    H: [B, heads, S, K, V] (kv) or [B, heads, S, V, K] (vk); M: [B, heads, S, K, K];
    h_init: [B, heads, state] or None (zeros).  Returns (out, final) with out
    shaped like H and final like h_init (None when not requested)."""
    H = _f32(H)
    M = _f32(M)
    h_init = _f32(h_init)
    B, heads, S = H.shape[:3]
    if layout == "kv":
        K, V = H.shape[3], H.shape[4]
        lay = 0
    elif layout == "vk":
        V, K = H.shape[3], H.shape[4]
        lay = 1
    else:
        raise ValueError(layout)
    assert M.shape == (B, heads, S, K, K), (M.shape, H.shape)
    if h_init is not None:
        assert h_init.shape == (B, heads) + H.shape[3:], (h_init.shape, H.shape)
    dirn = {"fwd": 0, "rev": 1}[direction]
    out = np.empty(H.shape, np.float64) if want_out else None
    fin = np.empty((B, heads) + H.shape[3:], np.float64) if want_final else None
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    p = lambda a, t: None if a is None else a.ctypes.data_as(t)  # noqa: E731
    used = _lib(variant).qla_oracle_cp_correct(p(H, f32p), p(M, f32p), p(h_init, f32p),
                                               p(out, f64p), p(fin, f64p), B * heads, S, K, V,
                                               lay, dirn, nthreads)
    if return_threads:
        return out, fin, used
    return out, fin
