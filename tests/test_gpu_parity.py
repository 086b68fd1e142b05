"""GPU parity: the CUDA path against the fp64 oracle on the same seeded inputs.

Bar (per output state): rel-L2 <= 1e-5 and max|err| <= 1e-4 * max|ref|; exact
when the reference state is all zero; bitwise on the exact-integer cases.
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi
from gpu_util import engine_supports, engines_under_test, run
from qla_check import assert_parity

pytestmark = pytest.mark.gpu

LAYOUTS = ("kv", "vk")
DIRS = ("fwd", "rev")
ENGINES = engines_under_test()


def skip_unsupported(engine, K, V):
    if not engine_supports(engine, K, V):
        pytest.skip(f"engine {engine} does not take K={K}, V={V}")


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("name", ["c0", "c1", "c2"])
def test_workloads(name, layout, direction, engine):
    c = qi.WORKLOADS[name]
    skip_unsupported(engine, c.K, c.V)
    H, M, h0 = qi.make_inputs(c, layout)
    ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
    got, fin = run(H, M, h0, layout, direction, engine=engine, final=True)
    assert_parity(got, ref, what=f"{name} {layout} {direction} {engine}")
    assert_parity(fin, rfin, what=f"{name} final")


@pytest.fixture(scope="module")
def large_inputs():
    c = qi.WORKLOADS["c3"]
    H, M, h0 = qi.make_inputs(c, "kv")
    return c, H, M, h0


def run_f32(H, M, h0, layout, direction, engine):
    """As gpu_util.run, but keeps the result in fp32 (the large workload's
    outputs are 2 GB in fp32)."""
    import torch
    import linear_attention_context_gb300 as qla
    from gpu_util import to_dev
    out = qla.cp_correct(to_dev(H), to_dev(M), to_dev(h0), layout=layout, direction=direction, engine=engine)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("direction", DIRS)
def test_large_workload_every_chain(large_inputs, direction):
    """B=4, 64 heads, K=V=256, S=32 at full size: every one of the 256 chains
    of every engine that takes K=256 (the automatic choice, 3xTF32 and FFMA)
    against the oracle, state by state.  The oracle runs once per block of
    chains and serves all engines."""
    c, H, M, h0 = large_inputs
    engines = [e for e in ("auto", "tc", "simt") if e == "auto" or (e in ENGINES and engine_supports(e, c.K, c.V))]
    got = {e: run_f32(H, M, h0, "kv", direction, e) for e in engines}
    n = c.chains
    flat = lambda a: a.reshape((1, n) + a.shape[2:])  # noqa: E731  chains in (b, h) order
    Hf, Mf, h0f = flat(H), flat(M), flat(h0)
    step = 32
    for c0 in range(0, n, step):
        sl = (slice(None), slice(c0, min(n, c0 + step)))
        ref, _ = oracle.cp_correct(Hf[sl], Mf[sl], h0f[sl], "kv", direction)
        for e in engines:
            assert_parity(flat(got[e])[sl], ref, what=f"c3 chains {c0}..{c0 + step - 1} {direction} {e}")


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("heads", qi.SWEEP_HEADS)
@pytest.mark.parametrize("S", qi.SWEEP_S)
def test_sweep_seq_and_scan(S, heads, layout, direction):
    c = qi.sweep_case(heads, S)
    H, M, h0 = qi.make_inputs(c, layout)
    ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
    for variant in ("seq", "scan"):
        got, fin = run(H, M, h0, layout, direction, variant=variant, final=True)
        assert_parity(got, ref, what=f"sweep S={S} heads={heads} {layout} {direction} {variant}")
        assert_parity(fin, rfin, what=f"sweep final {variant}")


EDGE = [
    # (B, heads, S, K, V, init)
    (1, 1, 1, 64, 64, True),
    (1, 1, 1, 128, 128, False),
    (1, 2, 2, 128, 128, False),
    (3, 5, 3, 32, 256, True),
    (2, 3, 5, 256, 32, True),
    (1, 7, 4, 96, 160, True),
    (2, 1, 9, 128, 64, True),
    (1, 3, 6, 256, 128, False),
    (1, 1, 3, 224, 96, True),
    (1, 2, 3, 128, 32, True),   # one column tile per chain
    (1, 1, 4, 128, 256, True),  # eight column tiles per chain
    (2, 2, 2, 256, 32, False),
]


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "B{}h{}S{}K{}V{}{}".format(*s[:5], "i" if s[5] else "z"))
def test_edge_shapes(shape, layout, direction, engine):
    B, nh, S, K, V, init = shape
    skip_unsupported(engine, K, V)
    c = qi.Case(B=B, heads=nh, S=S, K=K, V=V, seed=77, m_kind="householder", h_scale=0.5,
                init_kind="gaussian" if init else "none")
    H, M, h0 = qi.make_inputs(c, layout)
    ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
    got, fin = run(H, M, h0, layout, direction, engine=engine, final=True)
    assert_parity(got, ref, what=f"edge {shape} {layout} {direction} {engine}")
    assert_parity(fin, rfin, what="edge final")
    # final state alone (no out)
    _, fin2 = run(H, M, h0, layout, direction, engine=engine, final=True, want_out=False)
    assert_parity(fin2, rfin, what="edge final only")


def test_more_chains_than_a_grid_y_dimension_holds():
    """70,000 chains (B = 70, heads = 1000): more units than the 65,535 a
    grid's y dimension takes, on the sequential variant and on the scan
    (140,000 units of two groups), through the one-dimensional grid."""
    c = qi.Case(B=70, heads=1000, S=2, K=32, V=32, seed=91, m_kind="householder", h_scale=0.5,
                init_kind="gaussian")
    H, M, h0 = qi.make_inputs(c, "kv")
    ref, rfin = oracle.cp_correct(H, M, h0, "kv", "fwd", want_final=True)
    for variant in ("seq", "scan"):
        got, fin = run(H, M, h0, "kv", "fwd", variant=variant, final=True)
        assert_parity(got, ref, what=f"70000 chains {variant}")
        assert_parity(fin, rfin, what=f"70000 chains {variant} final")


# Magnitudes far from 1: the 3xTF32 split keeps the hi and lo parts inside
# fp32's exponent range, so tiny and huge states and matrices must come through
# with the same relative accuracy.
RANGES = [
    # (m_scale, h_scale, init_scale): M = m_scale * orthogonal
    (0.99, 1e-20, 1e-20),  # tiny states
    (0.99, 1e12, 1e12),    # huge states
    (1e-9, 1.0, 1.0),      # tiny propagation matrices
    (3e5, 1.0, 1.0),       # huge propagation entries
    (0.99, 0.0, 1.0),      # no local states: pure propagation of h_init
]


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("rng", RANGES, ids=lambda r: "m{:g}_h{:g}_i{:g}".format(*r))
def test_dynamic_range(rng, direction, engine):
    m_scale, h_scale, init_scale = rng
    c = qi.Case(B=1, heads=2, S=4, K=128, V=64, seed=91, m_kind="orthogonal", m_scale=m_scale,
                h_scale=h_scale, init_kind="gaussian", init_scale=init_scale)
    for layout in LAYOUTS:
        H, M, h0 = qi.make_inputs(c, layout)
        ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
        got, fin = run(H, M, h0, layout, direction, engine=engine, final=True)
        assert np.isfinite(got).all() and np.isfinite(fin).all()
        assert_parity(got, ref, what=f"range {rng} {layout} {direction} {engine}")
        assert_parity(fin, rfin, what=f"range {rng} final")


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("direction", DIRS)
def test_rows_of_different_magnitude(direction, engine):
    """M = diag(d) Q with d spanning 10^-6 .. 10^6 (and rows of zeros): one
    scale per matrix must serve rows twelve decades apart."""
    c = qi.Case(B=1, heads=2, S=5, K=128, V=64, seed=92, m_kind="orthogonal", m_scale=1.0, h_scale=1.0,
                init_kind="gaussian")
    d = np.logspace(-6, 6, 128)
    d[::17] = 0.0
    for layout in LAYOUTS:
        H, M, h0 = qi.make_inputs(c, layout)
        M = np.ascontiguousarray(M * d[:, None]).astype(np.float32)
        ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
        got, fin = run(H, M, h0, layout, direction, engine=engine, final=True)
        assert_parity(got, ref, what=f"row magnitudes {layout} {direction} {engine}")
        assert_parity(fin, rfin, what="row magnitudes final")


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_in_place_matches_separate_output(layout, direction, engine):
    c = qi.WORKLOADS["c1"].with_(heads=4)
    H, M, h0 = qi.make_inputs(c, layout)
    ref, _ = oracle.cp_correct(H, M, h0, layout, direction)
    got, _ = run(H, M, h0, layout, direction, engine=engine, in_place=True)
    assert_parity(got, ref, what=f"in place {layout} {direction} {engine}")
    sep, _ = run(H, M, h0, layout, direction, engine=engine)
    assert np.array_equal(got, sep)


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("K,V", [(128, 128), (256, 64), (64, 32)])
def test_integer_exact_bitwise(K, V, layout, direction, engine):
    skip_unsupported(engine, K, V)
    c = qi.Case(B=1, heads=3, S=8, K=K, V=V, seed=5, m_kind="signed_perm", h_kind="small_int",
                init_kind="small_int")
    H, M, h0 = qi.make_inputs(c, layout)
    ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
    got, fin = run(H, M, h0, layout, direction, engine=engine, final=True)
    assert np.array_equal(got, ref)
    assert np.array_equal(fin, rfin)


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("group", [1, 2, 3, 7, 10])
def test_scan_groups_ragged(group, direction):
    c = qi.sweep_case(heads=2, S=10)
    for layout in LAYOUTS:
        H, M, h0 = qi.make_inputs(c, layout)
        ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
        got, fin = run(H, M, h0, layout, direction, variant="scan", scan_group=group, final=True)
        assert_parity(got, ref, what=f"scan group {group} {layout} {direction}")
        assert_parity(fin, rfin, what="scan final")


@pytest.mark.parametrize("direction", DIRS)
def test_scan_integer_exact(direction):
    c = qi.Case(B=1, heads=2, S=12, K=128, V=64, seed=8, m_kind="signed_perm", h_kind="small_int",
                init_kind="small_int")
    for layout in LAYOUTS:
        H, M, h0 = qi.make_inputs(c, layout)
        ref, _ = oracle.cp_correct(H, M, h0, layout, direction)
        got, _ = run(H, M, h0, layout, direction, variant="scan", scan_group=4)
        assert np.array_equal(got, ref)


def test_concurrent_scans_from_two_host_threads():
    """The scan's side stream and events are shared by a device's callers:
    two host threads running scans on their own streams must both be right."""
    import threading

    import torch

    import linear_attention_context_gb300 as qla
    dev = torch.device("cuda:0")
    c = qi.sweep_case(2, 32)
    cases = []
    for layout, direction in (("kv", "fwd"), ("vk", "rev")):
        H, M, h0 = qi.make_inputs(c, layout)
        ref, _ = oracle.cp_correct(H, M, h0, layout, direction)
        cases.append((layout, direction, torch.from_numpy(H).to(dev), torch.from_numpy(M).to(dev),
                      torch.from_numpy(h0).to(dev), ref))
    results, errors = {}, []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            layout, direction, Hd, Md, h0d, _ = cases[i]
            s = torch.cuda.Stream(dev)
            outs = []
            for _ in range(20):
                outs.append(qla.cp_correct(Hd, Md, h0d, layout=layout, direction=direction, variant="scan",
                                           stream=s))
            s.synchronize()
            results[i] = [o.cpu().numpy().astype(np.float64) for o in outs]
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (layout, direction, *_, ref) in enumerate(cases):
        for k, got in enumerate(results[i]):
            assert_parity(got, ref, what=f"thread {i} call {k} {layout} {direction}")
    assert qla.device_status() == 0


def test_process_wide_variant_override():
    """qla_set_variant forces the variant of every automatic choice (the plain
    entry point included); QLA_VARIANT sets its initial value."""
    import os
    import subprocess
    import sys

    import torch

    import linear_attention_context_gb300 as qla
    assert qla.resolve(1, 32, 8, 128, 128, "kv")[0] == "seq"
    c = qi.sweep_case(2, 8)
    H, M, h0 = qi.make_inputs(c, "vk")
    ref, _ = oracle.cp_correct(H, M, h0, "vk", "rev")
    try:
        qla.set_variant("scan")
        assert qla.resolve(1, 32, 8, 128, 128, "kv")[0] == "scan"
        got = qla.cp_correct(torch.from_numpy(H).cuda(), torch.from_numpy(M).cuda(), torch.from_numpy(h0).cuda(),
                             layout="vk", direction="rev")
        torch.cuda.synchronize()
        assert_parity(got.cpu().numpy().astype(np.float64), ref, what="forced scan")
    finally:
        qla.set_variant("auto")
    assert qla.resolve(1, 32, 8, 128, 128, "kv")[0] == "seq"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = "import linear_attention_context_gb300 as q; print(q.resolve(1, 32, 8, 128, 128, 'kv')[0])"
    env = dict(os.environ, QLA_VARIANT="scan")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "scan"


@pytest.mark.parametrize("engine", ENGINES)
def test_long_norm_preserving_chain(engine):
    """S = 128 with orthogonal M (no decay): the worst case for the tensor-core
    engines' accumulators, which round toward zero (a coherent shrink of about
    4e-8 per step); still inside the bar."""
    if not engine_supports(engine, 128, 128):
        pytest.skip(f"engine {engine} does not take K=128")
    c = qi.Case(B=1, heads=2, S=128, K=128, V=128, seed=11, m_kind="orthogonal", m_scale=1.0, h_scale=0.1,
                init_kind="gaussian", init_scale=0.1)
    H, M, h0 = qi.make_inputs(c, "kv")
    for direction in DIRS:
        ref, _ = oracle.cp_correct(H, M, h0, "kv", direction)
        got, _ = run(H, M, h0, "kv", direction, engine=engine, variant="seq")
        assert_parity(got, ref, what=f"S=128 orthogonal {direction} {engine}")


def test_ffma_engine_on_a_very_long_chain():
    """S = 512 with orthogonal M: the FFMA engine (round-to-nearest fp32
    accumulation) stays inside the bar where the tensor-core engines' drift
    does not (1.3e-5 at S = 256, 2.6e-5 at S = 512, measured)."""
    c = qi.Case(B=1, heads=1, S=512, K=128, V=64, seed=13, m_kind="orthogonal", m_scale=1.0, h_scale=0.1,
                init_kind="gaussian", init_scale=0.1)
    H, M, h0 = qi.make_inputs(c, "vk")
    ref, _ = oracle.cp_correct(H, M, h0, "vk", "fwd")
    got, _ = run(H, M, h0, "vk", "fwd", engine="simt", variant="seq")
    assert_parity(got, ref, what="S=512 orthogonal simt")


@pytest.mark.parametrize("layout,direction", [("kv", "fwd"), ("vk", "rev"), ("vk", "fwd"), ("kv", "rev")])
def test_plain_entry_point_through_the_c_abi(layout, direction):
    """qla_cp_correct, the entry point with the library's default choices,
    called directly through ctypes on the 32-head workload (and in place)."""
    import ctypes

    import torch

    import linear_attention_context_gb300 as qla
    from gpu_util import to_dev
    c = qi.WORKLOADS["c1" if direction == "fwd" else "c2"]
    H, M, h0 = qi.make_inputs(c, layout)
    ref, _ = oracle.cp_correct(H, M, h0, layout, direction)
    Hd, Md, h0d = to_dev(H), to_dev(M), to_dev(h0)
    out = torch.full_like(Hd, float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    lay, dirn = qla.LAYOUTS[layout], qla.DIRECTIONS[direction]
    rc = qla.lib().qla_cp_correct(p(Hd), p(Md), p(h0d), p(out), c.B, c.heads, c.S, c.K, c.V, lay, dirn, stream)
    assert rc == 0, qla.last_error()
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy().astype(np.float64), ref, what=f"qla_cp_correct {layout} {direction}")
    # in place (out == H), and a NULL h_init meaning zeros
    rc = qla.lib().qla_cp_correct(p(Hd), p(Md), None, p(Hd), c.B, c.heads, c.S, c.K, c.V, lay, dirn, stream)
    assert rc == 0, qla.last_error()
    torch.cuda.synchronize()
    ref0, _ = oracle.cp_correct(H, M, None, layout, direction)
    assert_parity(Hd.cpu().numpy().astype(np.float64), ref0, what=f"qla_cp_correct in place {layout} {direction}")


@pytest.mark.parametrize("K,S", [(128, 160), (128, 256), (128, 512), (256, 48), (256, 64), (256, 128)])
def test_automatic_choice_keeps_the_bar_on_long_undecayed_chains(K, S):
    """Orthogonal M without decay is the worst case for the tensor core's
    round-toward-zero accumulation (a coherent shrink every step).  The
    automatic engine takes the 3xTF32 engine up to 160 segments at K = 128
    and 48 at K = 256 and the FFMA engine beyond; either way the results stay
    inside the bar, in both variants and both directions."""
    import linear_attention_context_gb300 as qla
    limit = 160 if K == 128 else 48
    _, engine = qla.resolve(1, 2, S, K, 64, "kv")
    assert engine == ("tc" if S <= limit else "simt")
    c = qi.Case(B=1, heads=2, S=S, K=K, V=64, seed=11, m_kind="orthogonal", m_scale=1.0, h_scale=0.1,
                init_kind="gaussian", init_scale=0.1)
    H, M, h0 = qi.make_inputs(c, "kv")
    for direction in DIRS:
        ref, rfin = oracle.cp_correct(H, M, h0, "kv", direction, want_final=True)
        for variant in ("auto", "seq", "scan"):
            got, fin = run(H, M, h0, "kv", direction, engine="auto", variant=variant, final=True)
            assert_parity(got, ref, what=f"auto engine K={K} S={S} {direction} {variant}")
            assert_parity(fin, rfin, what=f"auto engine final K={K} S={S} {direction} {variant}")


def _scan_model(S, G, chains, K, V, sms):
    # the documented cost models of the two variants (us); waves of one-CTA-per-SM phases
    w = lambda n: -(-n // sms)  # noqa: E731
    Ls = -(-S // G)
    Gr = -(-S // Ls)
    return (4.74 + 1.96 * Ls * w(chains * Gr * ((K + V) // 32)) + 2.01 * Gr * w(chains * (V // 32))
            + 1.24 * Ls * w(chains * Gr * (V // 32)))


@pytest.mark.parametrize("heads,S", [(1, 32), (1, 128), (2, 128), (4, 32), (4, 128), (8, 64), (8, 128),
                                     (16, 128), (32, 8), (32, 128), (4, 16), (1, 3)])
def test_automatic_scan_groups_and_variant_follow_the_cost_models(heads, S):
    """The automatic group count (read back from the scratch size) is the cost
    model's fastest G up to round(sqrt(2 S)), and the automatic variant is the
    scan exactly where that model is below 0.95 of the sequential kernel's."""
    import math
    import torch
    import linear_attention_context_gb300 as qla
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    K = V = 128
    G0 = max(1, round(math.sqrt(2 * S)))
    cands = [G for G in range(1, min(G0, S) + 1) if -(-S // -(-S // G)) == G]
    best = min(cands, key=lambda G: (_scan_model(S, G, heads, K, V, sms), G))
    per_group = heads * (K * K + 2 * K * V) * 4
    assert qla.scan_workspace_bytes(1, heads, S, K, V) == best * per_group
    seq = 4.7 + 1.62 * (S - 1) * -(-(heads * (V // 32)) // sms)
    want = "scan" if S >= 2 and _scan_model(S, best, heads, K, V, sms) < 0.95 * seq else "seq"
    assert qla.resolve(1, heads, S, K, V)[0] == want
