"""Programmatic dependent launch (qla_set_dependent_launch), after xuesongtap,
"PTX 内存一致性", section on PDL: a trigger lets the dependent grid start,
but only griddepcontrol.wait makes the previous grid's writes visible.

A test producer lets its dependents start at once and writes one input of the
correction only after a delay; the correction, launched right after it as a
dependent, is then resident while that input still holds stale bytes (NaN, or
all-zero offsets).  The results must equal the oracle's on the produced
values, for every engine, each input in turn (H, M, h_init, the
variable-length offsets), and inside a CUDA graph, where the launch becomes a
programmatic edge.
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi
from gpu_util import engine_supports, engines_under_test, to_dev
from qla_check import assert_parity

pytestmark = pytest.mark.gpu

ENGINES = engines_under_test()
DELAY_US = 300


@pytest.fixture
def qla_dependent():
    import linear_attention_context_gb300 as qla
    qla.set_dependent_launch(True)
    yield qla
    qla.set_dependent_launch(False)


def _inputs(layout="kv"):
    c = qi.Case(B=1, heads=4, S=8, K=128, V=128, seed=23, h_scale=0.1, init_scale=0.1)
    return qi.make_inputs(c, layout)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("produced", ["H", "M", "h_init"])
@pytest.mark.parametrize("layout, direction", [("kv", "fwd"), ("vk", "rev")])
def test_dependent_reads_what_the_producer_wrote(qla_dependent, engine, produced, layout, direction):
    import torch
    qla = qla_dependent
    if not engine_supports(engine, 128, 128):
        pytest.skip(f"engine {engine} does not take K=128")
    H, M, h0 = _inputs(layout)
    ref, _ = oracle.cp_correct(H, M, h0, layout, direction)
    dev = {"H": to_dev(H), "M": to_dev(M), "h_init": to_dev(h0)}
    src = dev[produced]
    dev[produced] = torch.full_like(src, float("nan"))  # what an early read would see
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        out = torch.empty_like(dev["H"])
        qla.selftest_dependent_producer(src, dev[produced], DELAY_US, stream)
        qla.cp_correct(dev["H"], dev["M"], dev["h_init"], out, layout=layout, direction=direction,
                       engine=engine, variant="seq", stream=stream)
    stream.synchronize()
    assert qla.device_status() == 0
    assert_parity(out.cpu().numpy().astype(np.float64), ref, what=f"dependent {produced} {engine}")


@pytest.mark.parametrize("engine", ENGINES)
def test_dependent_reads_produced_offsets(qla_dependent, engine):
    import torch
    qla = qla_dependent
    if not engine_supports(engine, 128, 128):
        pytest.skip(f"engine {engine} does not take K=128")
    H, M, h0, cu = qi.make_varlen_inputs([3, 0, 5, 8], 2, 128, 128, seed=29, h_scale=0.1, init_scale=0.1)
    ref, rfin = oracle.cp_correct_varlen(H, M, h0, cu, "kv", "fwd")
    Hd, Md, h0d = to_dev(H), to_dev(M), to_dev(h0)
    # 5 offsets are 20 bytes: the producer copies whole 16-byte words, so pad both sides to 8.
    cu_src = torch.zeros(8, dtype=torch.int32, device="cuda:0")
    cu_src[:len(cu)] = torch.from_numpy(cu.astype(np.int32)).to("cuda:0")
    cu_dst = torch.zeros(8, dtype=torch.int32, device="cuda:0")  # stale: every sequence empty
    fin = torch.empty((len(cu) - 1, 2, 128, 128), device="cuda:0")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        out = torch.zeros_like(Hd)
        qla.selftest_dependent_producer(cu_src, cu_dst, DELAY_US, stream)
        qla.cp_correct_varlen(Hd, Md, cu_dst[:len(cu)], h0d, out, layout="kv", direction="fwd",
                              final_state=fin, engine=engine, stream=stream)
    stream.synchronize()
    assert qla.device_status() == 0
    assert_parity(out.cpu().numpy().astype(np.float64), ref, what=f"dependent offsets {engine}")
    assert_parity(fin.cpu().numpy().astype(np.float64), rfin, what=f"dependent offsets final {engine}")


def test_dependent_launch_in_a_graph(qla_dependent):
    """Producer and correction captured together; each replay copies a new H."""
    import torch
    qla = qla_dependent
    H, M, h0 = _inputs()
    H2 = (H[:, :, ::-1] * np.float32(0.5)).copy()  # a second, different H
    refs = [oracle.cp_correct(x, M, h0, "kv", "fwd")[0] for x in (H, H2)]
    srcs = [to_dev(H), to_dev(H2)]
    src = torch.empty_like(srcs[0])
    Hd = torch.full_like(src, float("nan"))
    Md, h0d = to_dev(M), to_dev(h0)
    out = torch.empty_like(Hd)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        # warm-up outside the capture (first-use set-up of the library and the kernels)
        src.copy_(srcs[0])
        qla.selftest_dependent_producer(src, Hd, DELAY_US, stream)
        qla.cp_correct(Hd, Md, h0d, out, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        qla.selftest_dependent_producer(src, Hd, DELAY_US, stream)
        qla.cp_correct(Hd, Md, h0d, out, stream=stream)
    for rep in range(4):
        with torch.cuda.stream(stream):
            src.copy_(srcs[rep % 2])
            Hd.fill_(float("nan"))
            g.replay()
        stream.synchronize()
        assert qla.device_status() == 0
        assert_parity(out.cpu().numpy().astype(np.float64), refs[rep % 2], what=f"graph replay {rep}")
