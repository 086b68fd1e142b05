"""Bounded waits: a stalled pipeline ends on its own and reports it.

qla_selftest_stalled_wait launches a warp-specialised engine with one
consumer waiting on a barrier that nothing arrives on.  Its wait gives up
after the given limit, the kernel records the event in the device status
word, every other role sees the abort, drains its copies in flight, frees
tensor memory and returns.  The context stays usable: a normal call after it
must still be correct.
"""
import ctypes
import time

import numpy as np
import pytest

import linear_attention_context_gb300 as qla
import oracle
import qla_inputs as qi
from qla_check import assert_parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("engine", ["tc"])
def test_stalled_wait_times_out_and_context_survives(engine):
    import torch
    dev = torch.device("cuda:0")
    c = qi.Case(B=1, heads=1, S=3, K=128, V=128, seed=3, h_scale=0.5, init_kind="none")
    H, M, _ = qi.make_inputs(c, "kv")
    Hd, Md = torch.from_numpy(H).to(dev), torch.from_numpy(M).to(dev)
    out = torch.zeros_like(Hd)
    assert qla.device_status() == 0  # clears any earlier word
    t0 = time.time()
    rc = qla.lib().qla_selftest_stalled_wait(ctypes.c_void_p(Hd.data_ptr()), ctypes.c_void_p(Md.data_ptr()),
                                              ctypes.c_void_p(out.data_ptr()), c.S, 20000, qla.ENGINES[engine],
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, qla.last_error()
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert qla.device_status() == 1
    assert qla.device_status() == 0  # read clears it
    assert elapsed < 5.0
    # the context is still usable and correct
    c2 = qi.WORKLOADS["c1"].with_(heads=2)
    H2, M2, h02 = qi.make_inputs(c2, "vk")
    got = qla.cp_correct(torch.from_numpy(H2).to(dev), torch.from_numpy(M2).to(dev), torch.from_numpy(h02).to(dev),
                         layout="vk", direction="rev", engine=engine)
    torch.cuda.synchronize()
    ref, _ = oracle.cp_correct(H2, M2, h02, "vk", "rev")
    assert_parity(got.cpu().numpy().astype(np.float64), ref, what=f"after stalled wait ({engine})")
    assert qla.device_status() == 0
