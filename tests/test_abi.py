"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments with the documented status before
it makes any CUDA call (so fake, never-dereferenced pointers are enough)."""
import ctypes
import os
import re

import pytest

import linear_attention_context_gb300 as qla
from linear_attention_context_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qla.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_build.library_path()):
        _build.build()
    return qla.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qla_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(qla.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_only_the_c_abi_is_exported(L):
    # hidden visibility keeps kernels and helpers out of the dynamic symbol table
    import subprocess
    r = subprocess.run(["nm", "-D", "--defined-only", _build.library_path()], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm unavailable")
    names = {ln.split()[-1] for ln in r.stdout.splitlines() if " T " in ln}
    qla_names = {n for n in names if n.startswith("qla_")}
    assert qla_names == set(declared_functions())


def test_version_and_status_strings(L):
    assert L.qla_version() == 100
    for code, name in qla.STATUS.items():
        assert L.qla_status_string(code).decode().startswith(name)
    assert L.qla_status_string(12345).decode() == "unknown status"


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def call(L, H=FAKE, M=FAKE + (1 << 32), h0=None, out=FAKE + (2 << 32), fin=None, B=1, heads=2, S=4, K=64,
         V=64, layout=0, direction=0, variant=0, engine=0, release=0, group=0):
    vp = ctypes.c_void_p
    return L.qla_cp_correct_ex(vp(H), vp(M), vp(h0), vp(out), vp(fin), B, heads, S, K, V, layout, direction,
                               variant, engine, release, group, None)


@pytest.mark.parametrize("kw,status", [
    (dict(H=None), -1), (dict(M=None), -1), (dict(out=None), -1),
    (dict(B=0), -1), (dict(heads=-1), -1), (dict(S=0), -1), (dict(K=0), -1),
    (dict(layout=2), -1), (dict(direction=-1), -1),
    (dict(variant=3), -1), (dict(engine=9), -1), (dict(engine=4), -1), (dict(engine=2), -1), (dict(release=7), -1),
    (dict(group=-1), -1),
    (dict(K=48), -2), (dict(V=288), -2), (dict(K=16), -2), (dict(V=100), -2),
    # one CTA per (chain, segment group, 32-column tile) must fit a 2^31 - 1 grid
    (dict(B=1 << 16, heads=1 << 10, S=16), -2),
    (dict(H=FAKE + 4), -3), (dict(M=FAKE + (1 << 32) + 8), -3), (dict(out=FAKE + (2 << 32) + 12), -3),
    (dict(h0=FAKE + (3 << 32) + 2), -3), (dict(fin=FAKE + (4 << 32) + 1), -3),
    # overlaps: out partially over H; M over H; h_init inside M; final over out
    (dict(out=FAKE + 16), -4), (dict(M=FAKE + 4096), -4), (dict(h0=FAKE + (1 << 32) + 64), -4),
    (dict(fin=FAKE + (2 << 32) + 1024), -4),
])
def test_argument_checks(L, kw, status):
    assert call(L, **kw) == status
    assert L.qla_last_error().decode() != ""


# The next three calls pass validation, so with a GPU present they would launch
# on the fake pointers; they run only where no GPU is visible.
no_gpu_only = pytest.mark.skipif("_has_gpu()", reason="would launch on fake pointers")


@no_gpu_only
def test_out_equal_to_H_passes_the_checks(L):
    # exact alias is the in-place mode: validation passes and the call stops
    # at the device probe
    assert call(L, out=FAKE) == -5


@no_gpu_only
def test_valid_call_without_gpu_reports_cuda_error(L):
    assert call(L) == -5
    assert "cuda" in L.qla_last_error().decode().lower()


@no_gpu_only
def test_more_chains_than_a_grid_y_dimension_pass_the_checks(L):
    # 70,000 chains: the grid is one-dimensional, so only its 2^31 - 1 CTAs bound them
    assert call(L, B=70, heads=1000, S=1) == -5
    assert call_varlen(L, N=70000, heads=1) == -5


@no_gpu_only
def test_final_state_only_is_accepted_by_checks(L):
    assert call(L, out=None, fin=FAKE + (4 << 32)) == -5


def test_scan_workspace_bytes(L):
    # chains * G * (K*K + 2*K*V) * 4 with G the groups actually formed
    assert L.qla_scan_workspace_bytes(1, 1, 128, 128, 128, 16) == 1 * 16 * (128 * 128 + 2 * 128 * 128) * 4
    assert L.qla_scan_workspace_bytes(2, 3, 10, 64, 32, 4) == 6 * 4 * (64 * 64 + 2 * 64 * 32) * 4
    # S = 10 with 3 groups: L = 4, so groups actually formed = 3
    assert L.qla_scan_workspace_bytes(1, 1, 10, 32, 32, 3) == 3 * (32 * 32 + 2 * 32 * 32) * 4
    assert L.qla_scan_workspace_bytes(0, 1, 10, 32, 32, 3) == 0


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def call_varlen(L, H=FAKE, M=FAKE + (1 << 32), h0=None, out=FAKE + (2 << 32), fin=None, cu=FAKE + (5 << 32), N=3,
                T=10, heads=2, K=64, V=64, layout=0, direction=0, engine=0):
    vp = ctypes.c_void_p
    return L.qla_cp_correct_varlen(vp(H), vp(M), vp(h0), vp(out), vp(fin), vp(cu), N, T, heads, K, V, layout,
                                   direction, engine, None)


@pytest.mark.parametrize("kw,status", [
    (dict(cu=None), -1), (dict(H=None), -1), (dict(M=None), -1), (dict(out=None), -1),
    (dict(N=0), -1), (dict(T=-1), -1), (dict(heads=0), -1), (dict(layout=3), -1), (dict(direction=2), -1),
    (dict(engine=4), -1), (dict(K=48), -2), (dict(V=300), -2), (dict(N=1 << 30, heads=2), -2),
    (dict(cu=FAKE + (5 << 32) + 2), -3), (dict(H=FAKE + 8), -3),
    (dict(cu=FAKE + 64), -4), (dict(out=FAKE + 4096), -4), (dict(h0=FAKE + (1 << 32) + 16), -4),
])
def test_varlen_argument_checks(L, kw, status):
    assert call_varlen(L, **kw) == status


def test_stalled_wait_selftest_argument_checks(L):
    vp = ctypes.c_void_p
    H, M, out = vp(FAKE), vp(FAKE + (1 << 32)), vp(FAKE + (2 << 32))
    assert L.qla_selftest_stalled_wait(H, M, out, 3, 1000, 1, None) == -1    # FFMA engine has no pipeline
    assert L.qla_selftest_stalled_wait(H, M, out, 3, 1000, 0, None) == -1    # automatic choice is not an engine
    assert L.qla_selftest_stalled_wait(H, M, out, 3, 1000, 2, None) == -1    # no engine 2
    assert L.qla_selftest_stalled_wait(H, M, out, 1, 1000, 3, None) == -1    # needs S >= 2
    assert L.qla_selftest_stalled_wait(H, M, out, 3, 0, 3, None) == -1       # limit outside [1, 10^7]


def call_varlen_ex(L, variant=0, max_segments=0, scan_group=0, **kw):
    args = dict(H=FAKE, M=FAKE + (1 << 32), h0=None, out=FAKE + (2 << 32), fin=None, cu=FAKE + (5 << 32), N=3,
                T=10, heads=2, K=64, V=64, layout=0, direction=0, engine=0)
    args.update(kw)
    vp = ctypes.c_void_p
    return L.qla_cp_correct_varlen_ex(vp(args["H"]), vp(args["M"]), vp(args["h0"]), vp(args["out"]),
                                      vp(args["fin"]), vp(args["cu"]), args["N"], args["T"], args["heads"],
                                      args["K"], args["V"], args["layout"], args["direction"], variant,
                                      args["engine"], max_segments, scan_group, None)


@pytest.mark.parametrize("kw,status", [
    (dict(variant=3), -1), (dict(variant=-1), -1), (dict(max_segments=-1), -1), (dict(max_segments=11), -1),
    (dict(scan_group=-2), -1), (dict(engine=4), -1), (dict(cu=None), -1), (dict(K=48), -2),
    (dict(cu=FAKE + (5 << 32) + 2), -3), (dict(out=FAKE + 4096), -4),
])
def test_varlen_ex_argument_checks(L, kw, status):
    assert call_varlen_ex(L, **kw) == status


def test_set_variant_checks(L):
    assert L.qla_set_variant(3) == -1
    assert L.qla_set_variant(-1) == -1
    assert L.qla_set_variant(1) == 0
    assert L.qla_set_variant(2) == 0
    assert L.qla_set_variant(0) == 0  # back to the automatic rule for the rest of the process


def test_set_dependent_launch_checks(L):
    assert L.qla_set_dependent_launch(2) == -1
    assert L.qla_set_dependent_launch(-1) == -1
    assert L.qla_set_dependent_launch(1) == 0
    assert L.qla_set_dependent_launch(0) == 0  # off again for the rest of the process


@pytest.mark.parametrize("src, dst, nbytes, delay, status", [
    (None, 0x1000, 16, 0, -1),         # NULL source
    (0x1000, None, 16, 0, -1),         # NULL destination
    (0x1000, 0x2000, 20, 0, -1),       # not a multiple of 16 bytes
    (0x1008, 0x2000, 16, 0, -3),       # misaligned
    (0x1000, 0x1010, 32, 0, -4),       # overlapping
    (0x1000, 0x2000, 16, -1, -1),      # negative delay
    (0x1000, 0x2000, 16, 100001, -1),  # delay above the bound
])
def test_dependent_producer_checks(L, src, dst, nbytes, delay, status):
    # (every case fails its host-side check before the device is touched)
    vp = ctypes.c_void_p
    assert L.qla_selftest_dependent_producer(None if src is None else vp(src), None if dst is None else vp(dst),
                                             nbytes, delay, None) == status


def call_local(L, k=FAKE, v=FAKE + (1 << 32), beta=FAKE + (2 << 32), g=FAKE + (3 << 32), H=FAKE + (4 << 32),
               M=FAKE + (5 << 32), B=1, heads=2, T=64, S=4, K=64, V=64, layout=0):
    vp = ctypes.c_void_p
    return L.qla_local_pass(vp(k), vp(v), vp(beta), vp(g), vp(H), vp(M), B, heads, T, S, K, V, layout, None)


@pytest.mark.parametrize("kw,status", [
    (dict(k=None), -1), (dict(v=None), -1), (dict(beta=None), -1), (dict(g=None), -1), (dict(H=None, M=None), -1),
    (dict(T=66), -1), (dict(S=0), -1), (dict(T=0), -1), (dict(B=0), -1), (dict(layout=2), -1),
    (dict(K=48), -2), (dict(V=288), -2), (dict(B=1 << 20, heads=1 << 10, T=1 << 12, S=1 << 12), -2),
    (dict(k=FAKE + 8), -3), (dict(v=FAKE + (1 << 32) + 2), -3), (dict(H=FAKE + (4 << 32) + 4), -3),
    (dict(M=FAKE + (5 << 32) + 8), -3), (dict(beta=FAKE + (2 << 32) + 2), -3), (dict(g=FAKE + (3 << 32) + 1), -3),
    # outputs over an input, or over each other
    (dict(H=FAKE + 64), -4), (dict(M=FAKE + (3 << 32) + 16), -4), (dict(M=FAKE + (4 << 32) + 4096), -4),
])
def test_local_pass_argument_checks(L, kw, status):
    assert call_local(L, **kw) == status
    assert L.qla_last_error().decode() != ""


@no_gpu_only
def test_local_pass_valid_call_without_gpu(L):
    assert call_local(L) == -5
    assert call_local(L, H=None) == -5 and call_local(L, M=None) == -5


def call_local_ex(L, split, T=64, S=4, **kw):
    vp = ctypes.c_void_p
    a = dict(k=FAKE, v=FAKE + (1 << 32), beta=FAKE + (2 << 32), g=FAKE + (3 << 32), H=FAKE + (4 << 32),
             M=FAKE + (5 << 32))
    a.update(kw)
    return L.qla_local_pass_ex(vp(a["k"]), vp(a["v"]), vp(a["beta"]), vp(a["g"]), vp(a["H"]), vp(a["M"]), 1, 2, T,
                               S, 64, 64, 0, split, None)


@pytest.mark.parametrize("split", [-1, 3, 32])
def test_local_pass_split_checks(L, split):
    # segment length T / S = 16: the split must be 0 or divide it
    assert call_local_ex(L, split) == -1
    assert "split" in L.qla_last_error().decode()


@no_gpu_only
def test_local_pass_valid_splits_without_gpu(L):
    for split in (0, 1, 2, 16):
        assert call_local_ex(L, split) == -5


@no_gpu_only
def test_automatic_scan_groups_without_a_device_take_the_step_count_rule(L):
    """Without a usable device the automatic group count is round(sqrt(2 S)),
    as many groups as the SM-aware rule ever takes (so the scratch size is an
    upper bound)."""
    import math
    for S in (2, 10, 32, 64, 128, 200):
        G = max(1, round(math.sqrt(2 * S)))
        Ls = -(-S // G)
        Gr = -(-S // Ls)
        assert L.qla_scan_workspace_bytes(1, 4, S, 128, 128, 0) == 4 * Gr * (128 * 128 + 2 * 128 * 128) * 4
