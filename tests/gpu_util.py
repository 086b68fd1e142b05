"""Helpers for the GPU tests: move seeded inputs to the device, call the C ABI
through the binding, and bring results back for comparison with the oracle."""
from __future__ import annotations

import os

import numpy as np

# Engines under test.  The tensor-core engine takes the shapes listed in
# tc_supports(); the FFMA engine takes every supported shape.
BUILT_ENGINES = ("simt", "tc")


def engines_under_test():
    env = os.environ.get("QLA_TEST_ENGINES")
    if env:
        return tuple(e for e in env.split(",") if e)
    return BUILT_ENGINES


def engine_supports(engine, K, V):
    if engine == "tc":
        return K in (128, 256) and V % 32 == 0
    return True


def dev():
    import torch
    return torch.device("cuda:0")


def to_dev(a):
    import torch
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def run(H, M, h0, layout, direction, engine="auto", variant="auto", in_place=False, final=False,
        scan_group=0, release="membar", want_out=True):
    """Runs the library on numpy inputs; returns (out, final) as fp64 numpy."""
    import torch
    import linear_attention_context_gb300 as qla
    Hd, Md, h0d = to_dev(H), to_dev(M), to_dev(h0)
    fin = torch.empty((H.shape[0], H.shape[1]) + H.shape[3:], dtype=torch.float32, device=dev()) if final else None
    out = Hd if in_place else None
    out = qla.cp_correct(Hd, Md, h0d, out, layout=layout, direction=direction, final_state=fin,
                         variant=variant, engine=engine, release=release, scan_group=scan_group,
                         want_out=want_out)
    torch.cuda.synchronize()
    o = None if out is None else out.cpu().numpy().astype(np.float64)
    f = None if fin is None else fin.cpu().numpy().astype(np.float64)
    return o, f


def run_varlen(H, M, h0, cu, layout, direction, engine, in_place=False, **kw):
    """Runs the variable-length form on numpy inputs (offsets `cu`, N + 1
    int32); returns (out, final) as numpy, after checking the device status
    word."""
    import torch
    import linear_attention_context_gb300 as qla
    Hd, Md, h0d = to_dev(H), to_dev(M), to_dev(h0)
    cud = to_dev(cu.astype(np.int32))
    N, heads = len(cu) - 1, H.shape[0]
    fin = torch.empty((N, heads) + H.shape[2:], device=dev())
    out = Hd if in_place else None
    out = qla.cp_correct_varlen(Hd, Md, cud, h0d, out, layout=layout, direction=direction, final_state=fin,
                                engine=engine, **kw)
    torch.cuda.synchronize()
    assert qla.device_status() == 0
    return out.cpu().numpy(), fin.cpu().numpy()
