"""GPU parity of the per-segment local pass (qla_local_pass) against the fp64
oracle (oracle.local_pass), and of the local pass chained into the state
correction.

Bar per output matrix (each H_i and each M_i): rel-L2 <= 1e-5 and
max|err| <= 1e-4 * max|ref|, as for the correction; bitwise on the exact
orthogonal-key case.
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi
from qla_check import assert_parity

pytestmark = pytest.mark.gpu


def dev():
    import torch
    return torch.device("cuda:0")


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def run_local(k, v, b, g, S, layout="kv", want_H=True, want_M=True):
    import torch
    import linear_attention_context_gb300 as qla
    H, M = qla.local_pass(to_dev(k), to_dev(v), to_dev(b), to_dev(g), S, layout=layout, want_H=want_H,
                          want_M=want_M)
    torch.cuda.synchronize()
    f = lambda t: None if t is None else t.cpu().numpy().astype(np.float64)  # noqa: E731
    return f(H), f(M)


def check_case(c, layout):
    k, v, b, g = qi.make_local_inputs(c)
    Hr, Mr = oracle.local_pass(k, v, b, g, c.S, layout)
    H, M = run_local(k, v, b, g, c.S, layout)
    assert_parity(H, Hr, what=f"local H {c} {layout}")
    assert_parity(M, Mr, what=f"local M {c} {layout}")


@pytest.mark.parametrize("layout", ["kv", "vk"])
def test_small_workload(layout):
    check_case(qi.LOCAL_WORKLOADS["l0"], layout)


def test_full_workload_every_segment():
    """32 heads, 32K tokens in 8 segments of 4K, K = V = 128: every H_i and
    M_i of every chain against the oracle."""
    check_case(qi.LOCAL_WORKLOADS["l1"], "kv")


EDGE = [
    # (B, heads, T, S, K, V): segment lengths 1, 33 and 100 are ragged against
    # the 32-token staging tile; K covers every rows-per-lane split
    (1, 1, 3, 3, 32, 32),
    (2, 3, 99, 3, 64, 224),
    (1, 2, 200, 2, 96, 64),
    (1, 2, 66, 2, 128, 32),
    (1, 1, 64, 2, 160, 96),
    (2, 1, 96, 3, 192, 128),
    (1, 1, 40, 1, 224, 32),
    (1, 2, 64, 2, 256, 256),
]


@pytest.mark.parametrize("layout", ["kv", "vk"])
@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "B{}h{}T{}S{}K{}V{}".format(*s))
def test_edge_shapes(shape, layout):
    B, nh, T, S, K, V = shape
    check_case(qi.LocalCase(B=B, heads=nh, T=T, S=S, K=K, V=V, seed=31), layout)


def test_strong_decays_rescale_the_state():
    """Decays of 0.6 - 0.8 per token: the log-decay falls by ~70 over a
    segment of 200 tokens, so the running scale is moved several times; M
    stays inside fp32's normal range."""
    c = qi.LocalCase(B=1, heads=2, T=400, S=2, K=64, V=64, seed=32, alpha_lo=0.6, alpha_hi=0.8)
    k, v, b, g = qi.make_local_inputs(c)
    assert g.reshape(2, 2, -1).sum(-1).max() < -40
    for layout in ("kv", "vk"):
        Hr, Mr = oracle.local_pass(k, v, b, g, c.S, layout)
        H, M = run_local(k, v, b, g, c.S, layout)
        assert_parity(H, Hr, what=f"strong decay H {layout}")
        assert_parity(M, Mr, what=f"strong decay M {layout}")


def test_growing_and_mixed_decays():
    """Log-decays of either sign (a_t in [0.5, 1.5]): the scale moves up as well
    as down."""
    c = qi.LocalCase(B=1, heads=2, T=128, S=2, K=64, V=32, seed=33, alpha_lo=0.5, alpha_hi=1.5, beta_hi=0.3)
    k, v, b, g = qi.make_local_inputs(c)
    Hr, Mr = oracle.local_pass(k, v, b, g, c.S)
    H, M = run_local(k, v, b, g, c.S)
    assert_parity(H, Hr, what="mixed decay H")
    assert_parity(M, Mr, what="mixed decay M")


@pytest.mark.parametrize("K,V", [(64, 64), (128, 32), (256, 64)])
def test_orthogonal_keys_bitwise(K, V):
    """Basis keys, b = 1, no decay, integer values: every operation is exact,
    so the kernel and the oracle agree bitwise."""
    rng = np.random.default_rng(K + V)
    S, L = 3, min(K, 40)
    T = S * L
    idx = np.concatenate([rng.permutation(K)[:L] for _ in range(S)])
    kf = np.zeros((1, 2, T, K), np.float32)
    kf[:, :, np.arange(T), idx] = 1.0
    vf = rng.integers(-8, 9, size=(1, 2, T, V)).astype(np.float32)
    k, v = qi.f32_to_bf16(kf), qi.f32_to_bf16(vf)
    b = np.ones((1, 2, T), np.float32)
    g = np.zeros((1, 2, T), np.float32)
    for layout in ("kv", "vk"):
        Hr, Mr = oracle.local_pass(k, v, b, g, S, layout)
        H, M = run_local(k, v, b, g, S, layout)
        assert np.array_equal(H, Hr) and np.array_equal(M, Mr)


def test_H_only_and_M_only():
    c = qi.LocalCase(B=1, heads=3, T=96, S=3, K=128, V=64, seed=34)
    k, v, b, g = qi.make_local_inputs(c)
    Hr, Mr = oracle.local_pass(k, v, b, g, c.S)
    H, M = run_local(k, v, b, g, c.S, want_M=False)
    assert M is None
    assert_parity(H, Hr, what="H only")
    H, M = run_local(k, v, b, g, c.S, want_H=False)
    assert H is None
    assert_parity(M, Mr, what="M only")


@pytest.mark.parametrize("graph", [False, True])
def test_local_pass_chained_into_the_correction(graph):
    """The local pass and the correction on one stream, the correction as a
    programmatic dependent (it launches while the local pass runs and reads H
    and M after its griddepcontrol.wait), plain and inside a CUDA graph that
    is replayed on changed inputs: the corrected states must match the
    oracle's correction of the oracle's local pass."""
    import torch
    import linear_attention_context_gb300 as qla
    c = qi.LOCAL_WORKLOADS["l1"].with_(heads=4, T=8192)
    layout = "kv"
    inputs = [qi.make_local_inputs(c.with_(seed=s)) for s in (41, 42)]
    h0 = qi.gaussian(c.chains, c.K * c.V, 43, qi.TENSOR_INIT, 0.1).reshape(1, c.heads, c.K, c.V)
    refs = []
    for k, v, b, g in inputs:
        Hr, Mr = oracle.local_pass(k, v, b, g, c.S, layout)
        refs.append(oracle.cp_correct(Hr.astype(np.float32), Mr.astype(np.float32), h0, layout, "fwd",
                                      want_final=True))
    dk, dv, db, dg = (to_dev(a) for a in inputs[0])
    h0d = to_dev(h0)
    H = torch.empty((1, c.heads, c.S, c.K, c.V), device=dev())
    M = torch.empty((1, c.heads, c.S, c.K, c.K), device=dev())
    out = torch.empty_like(H)
    fin = torch.empty((1, c.heads, c.K, c.V), device=dev())
    s = torch.cuda.Stream(dev())

    def pair():
        qla.local_pass(dk, dv, db, dg, c.S, H, M, layout=layout, stream=s)
        qla.cp_correct(H, M, h0d, out, layout=layout, final_state=fin, variant="seq", stream=s)

    qla.set_dependent_launch(True)
    try:
        if graph:
            pair()  # first calls outside the capture (device set-up)
            s.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(gr, stream=s):
                    pair()
        for rep in range(2):
            for t, a in zip((dk, dv, db, dg), inputs[rep]):
                t.copy_(torch.from_numpy(np.ascontiguousarray(a)))
            torch.cuda.synchronize()
            if graph:
                with torch.cuda.stream(s):
                    gr.replay()
            else:
                pair()
            s.synchronize()
            ref, rfin = refs[rep]
            assert_parity(out.cpu().numpy().astype(np.float64), ref, what=f"chained out rep {rep} graph {graph}")
            assert_parity(fin.cpu().numpy().astype(np.float64), rfin, what=f"chained final rep {rep}")
    finally:
        qla.set_dependent_launch(False)
    assert qla.device_status() == 0


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("layout", ["kv", "vk"])
def test_sub_segment_split(split, layout):
    """Each segment run as `split` sub-segments whose maps the correction
    kernels compose (M_i = product of the sub-segment M's, H_i = their
    recurrence from zero): the same H and M as the oracle, for both parts, H
    alone and M alone."""
    import torch
    import linear_attention_context_gb300 as qla
    c = qi.LocalCase(B=1, heads=3, T=1024, S=2, K=128, V=64, seed=35)
    k, v, b, g = qi.make_local_inputs(c)
    Hr, Mr = oracle.local_pass(k, v, b, g, c.S, layout)
    dk, dv, db, dg = (to_dev(a) for a in (k, v, b, g))
    for want_H, want_M in ((True, True), (True, False), (False, True)):
        H, M = qla.local_pass(dk, dv, db, dg, c.S, layout=layout, want_H=want_H, want_M=want_M, split=split)
        torch.cuda.synchronize()
        if want_H:
            assert_parity(H.cpu().numpy().astype(np.float64), Hr, what=f"split {split} H {layout}")
        if want_M:
            assert_parity(M.cpu().numpy().astype(np.float64), Mr, what=f"split {split} M {layout}")


@pytest.mark.parametrize("K,V", [(64, 32), (256, 64), (96, 160)])
def test_sub_segment_split_other_widths(K, V):
    """The composition runs on the 3xTF32 engine (K = 128, 256) or the FFMA
    engine (other K)."""
    import torch
    import linear_attention_context_gb300 as qla
    c = qi.LocalCase(B=1, heads=2, T=512, S=2, K=K, V=V, seed=36)
    k, v, b, g = qi.make_local_inputs(c)
    Hr, Mr = oracle.local_pass(k, v, b, g, c.S)
    H, M = qla.local_pass(*(to_dev(a) for a in (k, v, b, g)), c.S, split=4)
    torch.cuda.synchronize()
    assert_parity(H.cpu().numpy().astype(np.float64), Hr, what=f"split K={K} V={V} H")
    assert_parity(M.cpu().numpy().astype(np.float64), Mr, what=f"split K={K} V={V} M")
