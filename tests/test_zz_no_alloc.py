"""The allocation-free scan entry point, qla_cp_correct_scan_static.

It serves callers that cannot allocate device memory during a call: code that
runs with a fixed device-memory budget handed out at start-up, and
latency-bound code that cannot afford the device synchronisation cudaMalloc
can cause.  It keeps the scan's scratch in a fixed array inside the library.

These tests call it through the C ABI and compare it with the fp64 oracle and
with the allocating scan (qla_cp_correct_ex with QLA_VARIANT_SCAN) within the
parity tolerance the other GPU tests use, on two calls in a row that share the
array; they cover a single segment (no scan phases) and check that a shape
needing more scratch than the array holds is refused before anything
launches.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import linear_attention_context_gb300 as qla
import oracle
import qla_inputs as qi
from qla_check import assert_parity

pytestmark = pytest.mark.gpu

LAY = {"kv": 0, "vk": 1}
DIR = {"fwd": 0, "rev": 1}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _device_case(c, layout):
    import torch
    H, M, h0 = qi.make_inputs(c, layout)
    dev = torch.device("cuda:0")
    Hd, Md, h0d = (torch.from_numpy(a).to(dev) for a in (H, M, h0))
    fin_shape = (c.B, c.heads) + H.shape[3:]
    return Hd, Md, h0d, fin_shape


def _call_static(Hd, Md, h0d, out, fin, c, layout, direction, group=0):
    return qla.lib().qla_cp_correct_scan_static(
        _ptr(Hd), _ptr(Md), _ptr(h0d), _ptr(out), _ptr(fin), c.B, c.heads, c.S, c.K, c.V, LAY[layout],
        DIR[direction], 0, 0, group, _stream())


def _call_alloc_scan(Hd, Md, h0d, out, fin, c, layout, direction, group=0):
    return qla.lib().qla_cp_correct_ex(
        _ptr(Hd), _ptr(Md), _ptr(h0d), _ptr(out), _ptr(fin), c.B, c.heads, c.S, c.K, c.V, LAY[layout],
        DIR[direction], 2, 0, 0, group, _stream())


def _host(t):
    return t.cpu().numpy().astype(np.float64)


def test_static_scan_matches_oracle_and_allocating_scan_on_two_calls():
    import torch
    cases = [(qi.sweep_case(heads=4, S=32), "kv", "fwd"), (qi.sweep_case(heads=4, S=32).with_(seed=9), "vk", "rev")]
    for c, _, _ in cases:
        assert qla.lib().qla_scan_workspace_bytes(c.B, c.heads, c.S, c.K, c.V, 0) <= qla.SCAN_STATIC_BYTES
    prepared = []
    for c, layout, direction in cases:
        Hd, Md, h0d, fin_shape = _device_case(c, layout)
        prepared.append((c, layout, direction, Hd, Md, h0d, fin_shape))
    # two calls in a row on one stream, sharing the fixed scratch array
    static_out = []
    for c, layout, direction, Hd, Md, h0d, fin_shape in prepared:
        out = torch.empty_like(Hd)
        fin = torch.empty(fin_shape, device=Hd.device)
        rc = _call_static(Hd, Md, h0d, out, fin, c, layout, direction)
        assert rc == 0, qla.last_error()
        static_out.append((out, fin))
    torch.cuda.synchronize()
    for (c, layout, direction, Hd, Md, h0d, fin_shape), (out, fin) in zip(prepared, static_out):
        H, M, h0 = qi.make_inputs(c, layout)
        ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
        assert_parity(_host(out), ref, what=f"static scan vs oracle {layout} {direction}")
        assert_parity(_host(fin), rfin, what=f"static scan final vs oracle {layout} {direction}")
        aref = torch.empty_like(Hd)
        afin = torch.empty(fin_shape, device=Hd.device)
        rc = _call_alloc_scan(Hd, Md, h0d, aref, afin, c, layout, direction)
        assert rc == 0, qla.last_error()
        torch.cuda.synchronize()
        assert_parity(_host(out), _host(aref), what=f"static scan vs allocating scan {layout} {direction}")
        assert_parity(_host(fin), _host(afin), what=f"static scan final vs allocating scan {layout} {direction}")


def test_static_entry_with_one_segment():
    """S = 1 has no scan phases: out[0] is h_init and the final state one step."""
    import torch
    c = qi.sweep_case(heads=4, S=1)
    for layout, direction in (("kv", "fwd"), ("vk", "rev")):
        Hd, Md, h0d, fin_shape = _device_case(c, layout)
        H, M, h0 = qi.make_inputs(c, layout)
        ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
        for _ in range(2):
            out = torch.full_like(Hd, float("nan"))
            fin = torch.full(fin_shape, float("nan"), device=Hd.device)
            rc = _call_static(Hd, Md, h0d, out, fin, c, layout, direction)
            assert rc == 0, qla.last_error()
            torch.cuda.synchronize()
            assert_parity(_host(out), ref, what=f"static S=1 {layout} {direction}")
            assert_parity(_host(fin), rfin, what=f"static S=1 final {layout} {direction}")


def test_static_scan_refuses_shapes_beyond_its_scratch():
    import torch
    c = qi.sweep_case(heads=8, S=128)
    need = qla.lib().qla_scan_workspace_bytes(c.B, c.heads, c.S, c.K, c.V, 0)
    assert need > qla.SCAN_STATIC_BYTES
    Hd, Md, h0d, fin_shape = _device_case(c, "kv")
    out = torch.full_like(Hd, 7.0)
    rc = _call_static(Hd, Md, h0d, out, None, c, "kv", "fwd")
    assert rc == -2
    msg = qla.last_error()
    assert str(need) in msg and str(qla.SCAN_STATIC_BYTES) in msg
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing launched
