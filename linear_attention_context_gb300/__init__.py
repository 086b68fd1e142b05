"""GB300 (sm_103a) context-parallel state-correction pass for chunked linear
attention.

This module is a thin binding of the C ABI in ``include/qla.h``: it checks and
marshals torch tensors (device memory and the current CUDA stream) and calls
the library.  Every step of the recurrence runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and the import fails loudly when the
library has not been built.

The recurrence (Antarx Memos, "一次 TileLang Warp Specialization 数值错误的定位与
修复", sections "从版本升级后的数值偏差开始" and "理解三个缓冲区"):
X_0 = h_init, X_{i+1} = propagate(M_i, X_i) + H_i, propagate = M X (kv) or
X M^T (vk) forward and with M^T in reverse; out[i] is the state entering
segment i in visiting order.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

LAYOUTS = {"kv": 0, "vk": 1}
DIRECTIONS = {"fwd": 0, "rev": 1}
VARIANTS = {"auto": 0, "seq": 1, "scan": 2}
ENGINES = {"auto": 0, "simt": 1, "tc": 3}
RELEASES = {"membar": 0, "proxy": 1, "delay": 2, "none": 3}

QLA_OK = 0
STATUS = {0: "QLA_OK", -1: "QLA_ERR_INVALID_ARG", -2: "QLA_ERR_UNSUPPORTED", -3: "QLA_ERR_ALIGNMENT",
          -4: "QLA_ERR_ALIAS", -5: "QLA_ERR_CUDA", -6: "QLA_ERR_ARCH", -7: "QLA_ERR_TIMEOUT"}

# Every function include/qla.h declares.
EXPORTS = ("qla_cp_correct", "qla_cp_correct_ex", "qla_cp_correct_varlen", "qla_cp_correct_varlen_ex",
           "qla_scan_workspace_bytes", "qla_set_variant", "qla_set_dependent_launch",
           "qla_resolve", "qla_status_string", "qla_last_error", "qla_device_status", "qla_selftest_stalled_wait",
           "qla_selftest_dependent_producer", "qla_cp_correct_scan_static", "qla_local_pass", "qla_local_pass_ex",
           "qla_version")

# Bytes of scratch the allocation-free scan entry point holds (QLA_SCAN_STATIC_BYTES).
SCAN_STATIC_BYTES = 8 << 20


class QlaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {detail}")


_LIB = None


def library_path() -> str:
    return _build.library_path()


def lib():
    """The loaded C library (ctypes).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with __graft_entry__.build() "
                              "(or python -m linear_attention_context_gb300._build)")
        L = ctypes.CDLL(path)
        vp, ci, cz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.qla_cp_correct.argtypes = [vp, vp, vp, vp] + [ci] * 7 + [vp]
        L.qla_cp_correct.restype = ci
        L.qla_cp_correct_ex.argtypes = [vp, vp, vp, vp, vp] + [ci] * 11 + [vp]
        L.qla_cp_correct_ex.restype = ci
        L.qla_cp_correct_varlen.argtypes = [vp, vp, vp, vp, vp, vp] + [ci] * 8 + [vp]
        L.qla_cp_correct_varlen.restype = ci
        L.qla_cp_correct_varlen_ex.argtypes = [vp, vp, vp, vp, vp, vp] + [ci] * 11 + [vp]
        L.qla_cp_correct_varlen_ex.restype = ci
        L.qla_set_variant.argtypes = [ci]
        L.qla_set_variant.restype = ci
        L.qla_set_dependent_launch.argtypes = [ci]
        L.qla_set_dependent_launch.restype = ci
        L.qla_selftest_dependent_producer.argtypes = [vp, vp, ctypes.c_size_t, ci, vp]
        L.qla_selftest_dependent_producer.restype = ci
        L.qla_scan_workspace_bytes.argtypes = [ci] * 6
        L.qla_scan_workspace_bytes.restype = cz
        L.qla_resolve.argtypes = [ci] * 6 + [ctypes.POINTER(ci), ctypes.POINTER(ci)]
        L.qla_resolve.restype = ci
        L.qla_status_string.argtypes = [ci]
        L.qla_status_string.restype = ctypes.c_char_p
        L.qla_last_error.argtypes = []
        L.qla_last_error.restype = ctypes.c_char_p
        L.qla_device_status.argtypes = [ctypes.POINTER(ci)]
        L.qla_device_status.restype = ci
        L.qla_selftest_stalled_wait.argtypes = [vp, vp, vp, ci, ci, ci, vp]
        L.qla_selftest_stalled_wait.restype = ci
        L.qla_cp_correct_scan_static.argtypes = [vp, vp, vp, vp, vp] + [ci] * 10 + [vp]
        L.qla_cp_correct_scan_static.restype = ci
        L.qla_local_pass.argtypes = [vp] * 6 + [ci] * 7 + [vp]
        L.qla_local_pass.restype = ci
        L.qla_local_pass_ex.argtypes = [vp] * 6 + [ci] * 8 + [vp]
        L.qla_local_pass_ex.restype = ci
        L.qla_version.argtypes = []
        L.qla_version.restype = ci
        _LIB = L
    return _LIB


def last_error() -> str:
    return lib().qla_last_error().decode()


def check(status: int):
    if status != QLA_OK:
        raise QlaError(status, last_error())
    return status


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _shape(H, M, layout):
    if H.dim() != 5:
        raise ValueError(f"H must be [B, heads, S, rows, cols], got {tuple(H.shape)}")
    B, nh, S, r, c = H.shape
    K, V = (r, c) if layout == "kv" else (c, r)
    if tuple(M.shape) != (B, nh, S, K, K):
        raise ValueError(f"M must be {(B, nh, S, K, K)}, got {tuple(M.shape)}")
    return B, nh, S, K, V


def _check_tensor(name, t, dev, shape=None):
    import torch
    if t is None:
        return
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def cp_correct(H, M, h_init=None, out=None, *, layout="kv", direction="fwd", final_state=None,
               variant="auto", engine="auto", release="membar", scan_group=0, stream=None,
               want_out=True):
    """Corrected states for every segment (see the module docstring).

    H: [B, heads, S, K, V] (kv) or [B, heads, S, V, K] (vk) float32 CUDA tensor;
    M: [B, heads, S, K, K]; h_init: [B, heads, state] or None for zeros;
    out: preallocated like H (may be H itself: in place), or None to allocate;
    final_state: preallocated [B, heads, state] to also receive the state after
    the last segment.  Runs on ``stream`` (default: torch's current stream) and
    returns ``out`` (None when ``want_out`` is False)."""
    import torch
    if layout not in LAYOUTS or direction not in DIRECTIONS:
        raise ValueError(f"layout {layout!r} / direction {direction!r}")
    B, nh, S, K, V = _shape(H, M, layout)
    dev = H.device
    if dev.type != "cuda":
        raise ValueError("H must be a CUDA tensor")
    st = tuple(H.shape[3:])
    _check_tensor("H", H, dev)
    _check_tensor("M", M, dev)
    _check_tensor("h_init", h_init, dev, (B, nh) + st)
    _check_tensor("final_state", final_state, dev, (B, nh) + st)
    if want_out and out is None:
        out = torch.empty_like(H)
    if out is not None:
        _check_tensor("out", out, dev, H.shape)
    with torch.cuda.device(dev):
        rc = lib().qla_cp_correct_ex(_ptr(H), _ptr(M), _ptr(h_init), _ptr(out), _ptr(final_state),
                                     B, nh, S, K, V, LAYOUTS[layout], DIRECTIONS[direction],
                                     VARIANTS[variant], ENGINES[engine], RELEASES[release],
                                     int(scan_group), _stream_handle(stream))
    check(rc)
    return out


def cp_correct_varlen(H, M, cu_seg, h_init=None, out=None, *, layout="kv", direction="fwd", final_state=None,
                      engine="auto", stream=None, want_out=True, variant="seq", max_segments=0, scan_group=0):
    """Variable-length form: N sequences packed along the segment axis.

    H: [heads, T, K, V] (kv) or [heads, T, V, K] (vk) float32 CUDA tensor;
    M: [heads, T, K, K]; cu_seg: int32 CUDA tensor of N + 1 offsets
    (sequence n owns segments cu_seg[n] .. cu_seg[n+1] - 1); h_init and
    final_state: [N, heads, state] or None; out like H (may be H), or None to
    allocate.  Returns ``out`` (None when ``want_out`` is False).  Offsets are
    checked on the device: invalid ones skip their chains and set bit 1 of the
    status word (``device_status()``).  ``variant`` "seq", "scan" or "auto";
    the scan sizes its groups from ``max_segments`` (an upper bound on every
    sequence's segment count, 0 = T) and ``scan_group`` (group count, 0 =
    automatic); a longer sequence is flagged like invalid offsets."""
    import torch
    if layout not in LAYOUTS or direction not in DIRECTIONS:
        raise ValueError(f"layout {layout!r} / direction {direction!r}")
    if H.dim() != 4:
        raise ValueError(f"H must be [heads, T, rows, cols], got {tuple(H.shape)}")
    heads, T, r, c = H.shape
    K, V = (r, c) if layout == "kv" else (c, r)
    if tuple(M.shape) != (heads, T, K, K):
        raise ValueError(f"M must be {(heads, T, K, K)}, got {tuple(M.shape)}")
    dev = H.device
    if dev.type != "cuda":
        raise ValueError("H must be a CUDA tensor")
    if cu_seg.dtype != torch.int32 or cu_seg.dim() != 1 or cu_seg.device != dev or not cu_seg.is_contiguous():
        raise ValueError("cu_seg must be a contiguous 1-D int32 tensor on H's device")
    N = cu_seg.numel() - 1
    st = tuple(H.shape[2:])
    _check_tensor("H", H, dev)
    _check_tensor("M", M, dev)
    _check_tensor("h_init", h_init, dev, (N, heads) + st)
    _check_tensor("final_state", final_state, dev, (N, heads) + st)
    if want_out and out is None:
        out = torch.empty_like(H)
    if out is not None:
        _check_tensor("out", out, dev, H.shape)
    with torch.cuda.device(dev):
        rc = lib().qla_cp_correct_varlen_ex(_ptr(H), _ptr(M), _ptr(h_init), _ptr(out), _ptr(final_state),
                                            _ptr(cu_seg), N, T, heads, K, V, LAYOUTS[layout],
                                            DIRECTIONS[direction], VARIANTS[variant], ENGINES[engine],
                                            int(max_segments), int(scan_group), _stream_handle(stream))
    check(rc)
    return out


def local_pass(k, v, beta, g, S, H=None, M=None, *, layout="kv", want_H=True, want_M=True, split=0, stream=None):
    """Per-segment local states H and propagation matrices M (the inputs of
    cp_correct) from token-level inputs, by the gated delta rule (include/qla.h,
    qla_local_pass).

    k: [B, heads, T, K] and v: [B, heads, T, V] CUDA tensors of dtype bfloat16
    (or int16 holding bf16 bit patterns); beta, g: [B, heads, T] float32 (write
    strengths, log-space decays); T a multiple of S.  H ([B, heads, S, K, V] kv
    or [B, heads, S, V, K] vk) and M ([B, heads, S, K, K]) float32 are
    allocated when not given.  ``split``: sub-segments per segment (0 =
    automatic; see qla_local_pass_ex).  Returns (H, M), None for a part not
    wanted."""
    import torch
    if layout not in LAYOUTS:
        raise ValueError(f"layout {layout!r}")
    if k.dim() != 4 or v.dim() != 4:
        raise ValueError("k and v must be [B, heads, T, K] and [B, heads, T, V]")
    B, nh, T, K = k.shape
    V = v.shape[3]
    dev = k.device
    if dev.type != "cuda":
        raise ValueError("k must be a CUDA tensor")
    for name, t in (("k", k), ("v", v)):
        if t.dtype not in (torch.bfloat16, torch.int16) or t.device != dev or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 (or int16) tensor on {dev}")
    if tuple(v.shape[:3]) != (B, nh, T):
        raise ValueError(f"v must be {(B, nh, T, V)}, got {tuple(v.shape)}")
    _check_tensor("beta", beta, dev, (B, nh, T))
    _check_tensor("g", g, dev, (B, nh, T))
    st = (K, V) if layout == "kv" else (V, K)
    if want_H and H is None:
        H = torch.empty((B, nh, S) + st, dtype=torch.float32, device=dev)
    if want_M and M is None:
        M = torch.empty((B, nh, S, K, K), dtype=torch.float32, device=dev)
    _check_tensor("H", H, dev, (B, nh, S) + st)
    _check_tensor("M", M, dev, (B, nh, S, K, K))
    with torch.cuda.device(dev):
        rc = lib().qla_local_pass_ex(_ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(H), _ptr(M), B, nh, T, S, K, V,
                                     LAYOUTS[layout], int(split), _stream_handle(stream))
    check(rc)
    return H, M


def set_variant(variant: str):
    """Process-wide override of the automatic variant choice ("auto", "seq" or
    "scan"); the initial value comes from the QLA_VARIANT environment variable."""
    check(lib().qla_set_variant(VARIANTS[variant]))


def set_dependent_launch(enable: bool):
    """Process-wide switch for programmatic dependent launch of the sequential
    variant's kernel; the initial value comes from the QLA_PDL environment
    variable."""
    check(lib().qla_set_dependent_launch(1 if enable else 0))


def selftest_dependent_producer(src, dst, delay_us: int, stream=None):
    """Copies src into dst (same-size contiguous CUDA tensors) with a test
    producer that lets its dependents start at once and copies only after
    `delay_us` microseconds."""
    if src.numel() * src.element_size() != dst.numel() * dst.element_size():
        raise ValueError("src and dst differ in size")
    check(lib().qla_selftest_dependent_producer(_ptr(src), _ptr(dst), src.numel() * src.element_size(),
                                                int(delay_us), _stream_handle(stream)))


def scan_workspace_bytes(B, heads, S, K, V, scan_group=0) -> int:
    return int(lib().qla_scan_workspace_bytes(B, heads, S, K, V, scan_group))


def resolve(B, heads, S, K, V, layout="kv"):
    """(variant, engine) names that 'auto' resolves to on the current device."""
    v, e = ctypes.c_int(), ctypes.c_int()
    check(lib().qla_resolve(B, heads, S, K, V, LAYOUTS[layout], ctypes.byref(v), ctypes.byref(e)))
    inv_v = {b: a for a, b in VARIANTS.items()}
    inv_e = {b: a for a, b in ENGINES.items()}
    return inv_v[v.value], inv_e[e.value]


def device_status() -> int:
    """Reads and clears the device status word (synchronises); 0 = no event,
    bit 0 a bounded wait gave up, bit 1 invalid variable-length offsets."""
    f = ctypes.c_int()
    rc = lib().qla_device_status(ctypes.byref(f))
    if rc not in (QLA_OK, -7, -1):
        check(rc)
    return f.value
