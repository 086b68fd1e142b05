"""fp64 oracle for the CP state-correction pass and for the per-segment local
pass that produces its inputs -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library's CUDA path never calls it and shares
no code with it.  The arithmetic lives in ``qla_oracle.c`` (the correction) and
``qla_local_oracle.c`` (the local pass); this module only marshals numpy arrays
through ctypes.
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
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.qla_oracle_local_pass.argtypes = [u16p, u16p, f32p, f32p, f64p, f64p, ctypes.c_int64,
                                              ci, ci, ci, ci, ci, ci]
        lib.qla_oracle_local_pass.restype = ci
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


def cp_correct_varlen(H, M, h_init, cu_seg, layout="kv", direction="fwd"):
    """Variable-length form: sequences of different segment counts packed
    along the segment axis.

    H: [heads, T, K, V] (kv) or [heads, T, V, K] (vk); M: [heads, T, K, K];
    cu_seg: N + 1 non-decreasing offsets with cu_seg[0] = 0 and cu_seg[N] = T,
    sequence n owning segments cu_seg[n] .. cu_seg[n+1] - 1; h_init: [N, heads,
    state] or None (zeros).  Each (sequence, head) chain is the fixed-length
    recurrence over its own segments, so this is cp_correct applied to each
    sequence's slice.  A sequence with no segment has no outputs and its final
    state is its initial state.  Returns (out shaped like H, final [N, heads,
    state]) in fp64."""
    H = _f32(H)
    M = _f32(M)
    h_init = _f32(h_init)
    cu = [int(x) for x in np.asarray(cu_seg).reshape(-1)]
    heads, T = H.shape[:2]
    state = H.shape[2:]
    N = len(cu) - 1
    assert N >= 0 and cu[0] == 0 and cu[-1] == T and all(a <= b for a, b in zip(cu, cu[1:])), cu
    assert M.shape[:2] == (heads, T)
    if h_init is not None:
        assert h_init.shape == (N, heads) + state, (h_init.shape, H.shape)
    out = np.zeros(H.shape, np.float64)
    fin = np.zeros((N, heads) + state, np.float64)
    for n in range(N):
        s0, s1 = cu[n], cu[n + 1]
        init = None if h_init is None else h_init[n:n + 1]
        if s1 == s0:
            if init is not None:
                fin[n] = init[0]
            continue
        o, f = cp_correct(H[None, :, s0:s1], M[None, :, s0:s1], init, layout, direction, want_final=True)
        out[:, s0:s1] = o[0]
        fin[n] = f[0]
    return out, fin


def local_pass(k, v, beta, g, S, layout="kv", want_H=True, want_M=True, nthreads=0, variant=""):
    """Per-segment local state H_i and propagation matrix M_i (gated delta
    rule, token by token, fp64); see qla_local_oracle.c.

    k: [B, heads, T, K] and v: [B, heads, T, V] bf16 bit patterns (uint16 or
    int16 arrays); beta, g: [B, heads, T] float32; T = S * L.  Returns (H, M):
    H [B, heads, S, K, V] (kv) or [B, heads, S, V, K] (vk), M [B, heads, S, K, K],
    fp64 (None where not wanted)."""
    k = np.ascontiguousarray(k).view(np.uint16)
    v = np.ascontiguousarray(v).view(np.uint16)
    beta = _f32(beta)
    g = _f32(g)
    B, heads, T, K = k.shape
    V = v.shape[3]
    assert v.shape[:3] == (B, heads, T) and beta.shape == (B, heads, T) and g.shape == (B, heads, T)
    assert S >= 1 and T % S == 0, (T, S)
    lay = {"kv": 0, "vk": 1}[layout]
    st = (K, V) if layout == "kv" else (V, K)
    H = np.empty((B, heads, S) + st, np.float64) if want_H else None
    M = np.empty((B, heads, S, K, K), np.float64) if want_M else None
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    p = lambda a, t: None if a is None else a.ctypes.data_as(t)  # noqa: E731
    _lib(variant).qla_oracle_local_pass(p(k, u16p), p(v, u16p), p(beta, f32p), p(g, f32p), p(H, f64p),
                                        p(M, f64p), B * heads, T, S, K, V, lay, nthreads)
    return H, M
