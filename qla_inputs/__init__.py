"""Seeded synthetic inputs for the CP state-correction pass.

Both the fp64 oracle and the CUDA path consume the fp32 arrays made here; this
module holds none of the recurrence's arithmetic.  The generators live in
``gen.c`` (SplitMix64 streams keyed by seed, tensor id and block index;
Box-Muller Gaussians; Householder, Haar-orthogonal and signed-permutation
matrices) and are loaded through ctypes.

Tensor shapes (all contiguous fp32):
  H      [B][heads][S][K][V] (kv layout) or [B][heads][S][V][K] (vk layout)
  M      [B][heads][S][K][K]
  h_init [B][heads][K][V] (kv) or [B][heads][V][K] (vk), or None for zeros
A block is one matrix: H block (b*heads + h)*S + i, M block likewise, h_init
block b*heads + h.  The layout does not change what is drawn, only how the flat
block is read.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field, replace

import numpy as np

from . import build as _build

TENSOR_H = 1
TENSOR_M = 2
TENSOR_INIT = 3
TENSOR_KEY = 4
TENSOR_VALUE = 5
TENSOR_BETA = 6
TENSOR_GATE = 7

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.library_path()
        if not os.path.exists(path):
            _build.build()
        lib = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        i64, u64, dbl, cint = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_int
        lib.qla_gen_gaussian.argtypes = [f32p, i64, i64, u64, u64, i64, dbl]
        lib.qla_gen_householder.argtypes = [f32p, i64, cint, u64, u64, i64, dbl, dbl]
        lib.qla_gen_orthogonal.argtypes = [f32p, i64, cint, u64, u64, i64, dbl]
        lib.qla_gen_signed_perm.argtypes = [f32p, i64, cint, u64, u64, i64]
        lib.qla_gen_small_int.argtypes = [f32p, i64, i64, u64, u64, i64, cint]
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.qla_gen_unit_bf16.argtypes = [u16p, i64, cint, u64, u64, i64]
        lib.qla_gen_gaussian_bf16.argtypes = [u16p, i64, i64, u64, u64, i64, dbl]
        lib.qla_gen_uniform.argtypes = [f32p, i64, i64, u64, u64, i64, dbl, dbl, cint]
        for fn in ("qla_gen_gaussian", "qla_gen_householder", "qla_gen_orthogonal",
                   "qla_gen_signed_perm", "qla_gen_small_int", "qla_gen_unit_bf16",
                   "qla_gen_gaussian_bf16", "qla_gen_uniform"):
            getattr(lib, fn).restype = None
        _LIB = lib
    return _LIB


def _ptr(a: np.ndarray):
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def gaussian(nblocks, block_elems, seed, tensor_id, scale=1.0, block0=0):
    out = np.empty(int(nblocks) * int(block_elems), np.float32)
    if out.size:
        _lib().qla_gen_gaussian(_ptr(out), nblocks, block_elems, seed, tensor_id, block0, scale)
    return out


def householder(nblocks, K, seed, tensor_id, gmin, gmax, block0=0):
    out = np.empty((int(nblocks), K, K), np.float32)
    if out.size:
        _lib().qla_gen_householder(_ptr(out), nblocks, K, seed, tensor_id, block0, gmin, gmax)
    return out


def orthogonal(nblocks, K, seed, tensor_id, scale=1.0, block0=0):
    out = np.empty((int(nblocks), K, K), np.float32)
    if out.size:
        _lib().qla_gen_orthogonal(_ptr(out), nblocks, K, seed, tensor_id, block0, scale)
    return out


def signed_perm(nblocks, K, seed, tensor_id, block0=0):
    out = np.empty((int(nblocks), K, K), np.float32)
    if out.size:
        _lib().qla_gen_signed_perm(_ptr(out), nblocks, K, seed, tensor_id, block0)
    return out


def small_int(nblocks, block_elems, seed, tensor_id, maxabs, block0=0):
    out = np.empty(int(nblocks) * int(block_elems), np.float32)
    if out.size:
        _lib().qla_gen_small_int(_ptr(out), nblocks, block_elems, seed, tensor_id, block0, maxabs)
    return out


@dataclass(frozen=True)
class Case:
    """One synthetic problem: shapes, the M family and the value scales."""
    B: int
    heads: int
    S: int
    K: int
    V: int
    seed: int
    m_kind: str = "householder"     # householder | orthogonal | signed_perm | identity | zero
    gmin: float = 0.9               # Householder gain range
    gmax: float = 1.0
    m_scale: float = 0.99           # orthogonal: M = m_scale * Q
    h_kind: str = "gaussian"        # gaussian | small_int | zero
    h_scale: float = 1.0
    init_kind: str = "gaussian"     # gaussian | small_int | none
    init_scale: float = 1.0
    int_max: int = 8
    tags: tuple = field(default=())

    @property
    def chains(self):
        return self.B * self.heads

    def with_(self, **kw):
        return replace(self, **kw)


def make_inputs(c: Case, layout: str = "kv", unit0: int = 0):
    """Returns (H, M, h_init) as numpy fp32 arrays shaped for ``layout``.

    h_init is None when ``c.init_kind == "none"`` (zero initial state).
    ``unit0`` is the index of this problem's first chain within a larger job
    of the same Case: the arrays are then exactly chains unit0 .. unit0 +
    B*heads - 1 of that job (the generator streams are keyed by block index),
    which is how a job is sharded across ranks."""
    n = c.chains
    KV = c.K * c.V
    b0 = unit0 * c.S
    if c.h_kind == "gaussian":
        H = gaussian(n * c.S, KV, c.seed, TENSOR_H, c.h_scale, block0=b0)
    elif c.h_kind == "small_int":
        H = small_int(n * c.S, KV, c.seed, TENSOR_H, c.int_max, block0=b0)
    elif c.h_kind == "zero":
        H = np.zeros(n * c.S * KV, np.float32)
    else:
        raise ValueError(c.h_kind)
    nm = n * c.S
    if c.m_kind == "householder":
        M = householder(nm, c.K, c.seed, TENSOR_M, c.gmin, c.gmax, block0=b0)
    elif c.m_kind == "orthogonal":
        M = orthogonal(nm, c.K, c.seed, TENSOR_M, c.m_scale, block0=b0)
    elif c.m_kind == "signed_perm":
        M = signed_perm(nm, c.K, c.seed, TENSOR_M, block0=b0)
    elif c.m_kind == "identity":
        M = np.broadcast_to(np.eye(c.K, dtype=np.float32), (nm, c.K, c.K)).copy()
    elif c.m_kind == "zero":
        M = np.zeros((nm, c.K, c.K), np.float32)
    else:
        raise ValueError(c.m_kind)
    if c.init_kind == "gaussian":
        h0 = gaussian(n, KV, c.seed, TENSOR_INIT, c.init_scale, block0=unit0)
    elif c.init_kind == "small_int":
        h0 = small_int(n, KV, c.seed, TENSOR_INIT, c.int_max, block0=unit0)
    elif c.init_kind == "none":
        h0 = None
    else:
        raise ValueError(c.init_kind)
    st = (c.K, c.V) if layout == "kv" else (c.V, c.K)
    H = H.reshape((c.B, c.heads, c.S) + st)
    M = M.reshape(c.B, c.heads, c.S, c.K, c.K)
    if h0 is not None:
        h0 = h0.reshape((c.B, c.heads) + st)
    return H, M, h0


# The workloads the tests and the benchmark run.  Sizes and value
# distributions follow the five problem statements: a small single-head
# Householder case; the 32-head K=V=128 S=8 forward (Householder) and reverse
# (0.99 * orthogonal) cases; the 4x64-head K=V=256 S=32 case; and the low
# batch*heads sweep that compares the sequential and scan variants.
WORKLOADS = {
    "c0": Case(B=1, heads=1, S=4, K=64, V=64, seed=0, m_kind="householder", gmin=0.9, gmax=1.0,
               h_scale=1.0, init_kind="none"),
    "c1": Case(B=1, heads=32, S=8, K=128, V=128, seed=1, m_kind="householder", gmin=0.9, gmax=1.0,
               h_scale=0.1, init_scale=0.1),
    "c2": Case(B=1, heads=32, S=8, K=128, V=128, seed=2, m_kind="orthogonal", m_scale=0.99,
               h_scale=0.1, init_scale=0.1),
    "c3": Case(B=4, heads=64, S=32, K=256, V=256, seed=3, m_kind="householder", gmin=0.95, gmax=1.0,
               h_scale=0.05, init_scale=0.05),
}


def sweep_case(heads: int, S: int) -> Case:
    """One point of the low batch*heads sweep (B=1, K=V=128, 0.99 * orthogonal M)."""
    return Case(B=1, heads=heads, S=S, K=128, V=128, seed=4, m_kind="orthogonal", m_scale=0.99,
                h_scale=0.1, init_scale=0.1)


SWEEP_HEADS = (1, 4, 32)
SWEEP_S = (2, 8, 32, 128)


def make_varlen_inputs(lengths, heads, K, V, seed, layout="kv", m_kind="householder", gmin=0.9, gmax=1.0,
                       m_scale=0.99, h_scale=1.0, init_scale=1.0, with_init=True):
    """Packed variable-length inputs: sequence n has lengths[n] segments.

    Returns (H [heads, T, state], M [heads, T, K, K], h_init [N, heads, state]
    or None, cu_seg int32 [N + 1]) as numpy arrays, state = (K, V) for kv and
    (V, K) for vk.  Blocks are keyed (seed, tensor, block index) like the
    fixed-length inputs; H and M blocks are numbered head-major (h * T + t)."""
    lengths = [int(x) for x in lengths]
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    N = len(lengths)
    KV = K * V
    H = gaussian(heads * T, KV, seed, TENSOR_H, h_scale)
    if m_kind == "householder":
        M = householder(heads * T, K, seed, TENSOR_M, gmin, gmax)
    elif m_kind == "orthogonal":
        M = orthogonal(heads * T, K, seed, TENSOR_M, m_scale)
    elif m_kind == "signed_perm":
        M = signed_perm(heads * T, K, seed, TENSOR_M)
    elif m_kind == "identity":
        M = np.broadcast_to(np.eye(K, dtype=np.float32), (heads * T, K, K)).copy()
    else:
        raise ValueError(m_kind)
    st = (K, V) if layout == "kv" else (V, K)
    H = H.reshape((heads, T) + st)
    M = M.reshape(heads, T, K, K)
    h0 = gaussian(N * heads, KV, seed, TENSOR_INIT, init_scale).reshape((N, heads) + st) if with_init else None
    return H, M, h0, cu


# ---------------------------------------------------------------- local pass inputs
#
# Token-level inputs of the per-segment local pass (gated delta rule):
#   k     [B][heads][T][K] bf16 (stored as int16 bit patterns): unit Gaussian directions
#   v     [B][heads][T][V] bf16: N(0,1) * v_scale
#   beta  [B][heads][T] fp32: U(beta_lo, beta_hi)
#   g     [B][heads][T] fp32: log of U(alpha_lo, alpha_hi), a log-space decay
# A k or v block is one token (chain * T + t); a beta or g block is one chain.

def _u16_ptr(a: np.ndarray):
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def unit_bf16(nblocks, dim, seed, tensor_id, block0=0):
    out = np.empty((int(nblocks), dim), np.uint16)
    if out.size:
        _lib().qla_gen_unit_bf16(_u16_ptr(out), nblocks, dim, seed, tensor_id, block0)
    return out


def gaussian_bf16(nblocks, block_elems, seed, tensor_id, scale=1.0, block0=0):
    out = np.empty((int(nblocks), int(block_elems)), np.uint16)
    if out.size:
        _lib().qla_gen_gaussian_bf16(_u16_ptr(out), nblocks, block_elems, seed, tensor_id, block0, scale)
    return out


def uniform(nblocks, block_elems, seed, tensor_id, lo, hi, log_space=False, block0=0):
    out = np.empty((int(nblocks), int(block_elems)), np.float32)
    if out.size:
        _lib().qla_gen_uniform(_ptr(out), nblocks, block_elems, seed, tensor_id, block0, lo, hi, int(log_space))
    return out


def bf16_to_f32(a):
    """Exact fp32 values of bf16 bit patterns (int16 or uint16 arrays)."""
    return (np.asarray(a).view(np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x):
    """bf16 bit patterns (int16) of fp32 values, rounded to nearest even."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16).view(np.int16)


@dataclass(frozen=True)
class LocalCase:
    """One synthetic local-pass problem: T tokens per chain in S segments."""
    B: int
    heads: int
    T: int
    S: int
    K: int
    V: int
    seed: int
    beta_lo: float = 0.0
    beta_hi: float = 1.0
    alpha_lo: float = 0.9
    alpha_hi: float = 1.0
    v_scale: float = 1.0

    @property
    def chains(self):
        return self.B * self.heads

    @property
    def L(self):
        return self.T // self.S

    def with_(self, **kw):
        return replace(self, **kw)


def make_local_inputs(c: LocalCase, unit0: int = 0):
    """Returns (k, v, beta, g): k, v int16 bf16 bit patterns [B, heads, T, K|V];
    beta, g float32 [B, heads, T].  ``unit0`` is this problem's first chain
    within a larger job of the same case (as for make_inputs)."""
    assert c.S >= 1 and c.T % c.S == 0
    n = c.chains
    k = unit_bf16(n * c.T, c.K, c.seed, TENSOR_KEY, block0=unit0 * c.T)
    v = gaussian_bf16(n * c.T, c.V, c.seed, TENSOR_VALUE, c.v_scale, block0=unit0 * c.T)
    beta = uniform(n, c.T, c.seed, TENSOR_BETA, c.beta_lo, c.beta_hi, block0=unit0)
    g = uniform(n, c.T, c.seed, TENSOR_GATE, c.alpha_lo, c.alpha_hi, log_space=True, block0=unit0)
    sh = (c.B, c.heads, c.T)
    return (k.view(np.int16).reshape(sh + (c.K,)), v.view(np.int16).reshape(sh + (c.V,)), beta.reshape(sh),
            g.reshape(sh))


# Local-pass workloads.  The pages give no token-level distributions; these
# keep each segment's propagation matrix well inside fp32's range and far from
# zero: a small single-head case with strong writes and decays, and the
# 32-head case of the correction workload (32K tokens in 8 segments of 4K,
# K = V = 128) with moderate writes (beta below 0.1) and decays near 1.
LOCAL_WORKLOADS = {
    "l0": LocalCase(B=1, heads=1, T=256, S=4, K=64, V=64, seed=20, beta_lo=0.0, beta_hi=1.0, alpha_lo=0.9,
                    alpha_hi=1.0),
    "l1": LocalCase(B=1, heads=32, T=32768, S=8, K=128, V=128, seed=21, beta_lo=0.0, beta_hi=0.1,
                    alpha_lo=0.999, alpha_hi=1.0),
}
