"""GPU parity of the variable-length form (qla_cp_correct_varlen and its
variant form) against the fp64 varlen oracle: sequences of different segment
counts, including empty and one-segment sequences, both layouts and
directions, every engine, with and without initial states, in place, the
sequential and the scan variant (group counts that leave empty and ragged
groups); and the device-side checks (a chain with invalid offsets, or longer
than the scan's bound, is flagged).
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi
from gpu_util import engine_supports, engines_under_test
from gpu_util import run_varlen as _run
from gpu_util import to_dev as _dev
from qla_check import assert_parity

pytestmark = pytest.mark.gpu

LENGTHS = [3, 0, 1, 8, 2, 0, 5, 13]


@pytest.mark.parametrize("engine", engines_under_test())
@pytest.mark.parametrize("direction", ["fwd", "rev"])
@pytest.mark.parametrize("layout", ["kv", "vk"])
@pytest.mark.parametrize("K", [64, 128])
def test_varlen_parity(K, layout, direction, engine):
    if not engine_supports(engine, K, K):
        pytest.skip(f"engine {engine} does not take K={K}")
    H, M, h0, cu = qi.make_varlen_inputs(LENGTHS, 3, K, K, seed=31, layout=layout, m_kind="orthogonal",
                                         h_scale=0.1, init_scale=0.1)
    ref, rfin = oracle.cp_correct_varlen(H, M, h0, cu, layout, direction)
    got, fin = _run(H, M, h0, cu, layout, direction, engine)
    assert_parity(got, ref, what=f"varlen K={K} {layout} {direction} {engine}")
    assert_parity(fin, rfin, what="varlen final")


@pytest.mark.parametrize("engine", engines_under_test())
def test_varlen_no_initial_state_in_place(engine):
    K = 128
    if not engine_supports(engine, K, K):
        pytest.skip(f"engine {engine} does not take K={K}")
    H, M, _, cu = qi.make_varlen_inputs([4, 1, 0, 6], 2, K, K, seed=5, with_init=False)
    ref, rfin = oracle.cp_correct_varlen(H, M, None, cu, "kv", "fwd")
    got, fin = _run(H, M, None, cu, "kv", "fwd", engine, in_place=True)
    assert_parity(got, ref, what=f"varlen in place {engine}")
    assert_parity(fin, rfin, what="varlen in place final")


@pytest.mark.parametrize("engine", engines_under_test())
def test_varlen_exact_integers(engine):
    """Signed-permutation M and small integers: bitwise equality."""
    K = 128
    if not engine_supports(engine, K, K):
        pytest.skip(f"engine {engine} does not take K={K}")
    lengths = [5, 0, 2, 9]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, heads = int(cu[-1]), 2
    rng = np.random.default_rng(7)
    H = rng.integers(-8, 9, (heads, T, K, K)).astype(np.float32)
    h0 = rng.integers(-8, 9, (len(lengths), heads, K, K)).astype(np.float32)
    _, M, _, _ = qi.make_varlen_inputs(lengths, heads, K, K, seed=7, m_kind="signed_perm", with_init=False)
    ref, rfin = oracle.cp_correct_varlen(H, M, h0, cu, "vk", "rev")
    got, fin = _run(H, M, h0, cu, "vk", "rev", engine)
    assert np.array_equal(got, ref.astype(np.float32)) and np.array_equal(fin, rfin.astype(np.float32))


@pytest.mark.parametrize("engine", engines_under_test())
def test_varlen_invalid_offsets_are_flagged_and_skipped(engine):
    import torch

    import linear_attention_context_gb300 as qla
    K = 128
    if not engine_supports(engine, K, K):
        pytest.skip(f"engine {engine} does not take K={K}")
    H, M, h0, cu = qi.make_varlen_inputs([2, 2, 1], 2, K, K, seed=3)
    bad = np.array([0, 2, 4, 9], np.int32)  # the last sequence runs past T = 5
    Hd, Md, h0d, cud = _dev(H), _dev(M), _dev(h0), _dev(bad)
    out = torch.full_like(Hd, 7.0)
    qla.cp_correct_varlen(Hd, Md, cud, h0d, out, engine=engine)
    flags = qla.device_status()
    assert flags == 2
    got = out.cpu().numpy()
    ref, _ = oracle.cp_correct_varlen(H[:, :4], M[:, :4], h0[:2], np.array([0, 2, 4]), "kv", "fwd")
    assert_parity(got[:, :4], ref, what="valid chains next to an invalid one")
    assert (got[:, 4] == 7.0).all()  # the skipped chain's segment is untouched
    assert qla.device_status() == 0  # the word was cleared


@pytest.mark.parametrize("engine", engines_under_test())
@pytest.mark.parametrize("direction", ["fwd", "rev"])
@pytest.mark.parametrize("layout", ["kv", "vk"])
@pytest.mark.parametrize("group,bound", [(1, 13), (2, 13), (3, 13), (5, 13), (4, 0), (13, 20)])
def test_varlen_scan_parity(group, bound, layout, direction, engine):
    """Scan variant: every chain is cut into `group` groups of ceil(bound / group)
    segments (bound 0 = T); sequences of 0 .. 13 segments leave empty and
    ragged groups."""
    K = 128
    if not engine_supports(engine, K, K):
        pytest.skip(f"engine {engine} does not take K={K}")
    H, M, h0, cu = qi.make_varlen_inputs(LENGTHS, 2, K, K, seed=41, layout=layout, m_kind="orthogonal",
                                         h_scale=0.1, init_scale=0.1)
    ref, rfin = oracle.cp_correct_varlen(H, M, h0, cu, layout, direction)
    got, fin = _run(H, M, h0, cu, layout, direction, engine, variant="scan", max_segments=bound,
                    scan_group=group)
    what = f"varlen scan G={group} bound={bound} {layout} {direction} {engine}"
    assert_parity(got, ref, what=what)
    assert_parity(fin, rfin, what=what + " final")


@pytest.mark.parametrize("engine", engines_under_test())
def test_varlen_scan_final_state_only_and_auto(engine):
    """Final state alone through the scan; and the automatic choice (long
    sequences, few chains) agrees with the oracle."""
    import torch

    import linear_attention_context_gb300 as qla
    K = 64 if engine == "simt" else 128
    if not engine_supports(engine, K, K):
        pytest.skip(f"engine {engine} does not take K={K}")
    lengths = [30, 0, 7]
    H, M, h0, cu = qi.make_varlen_inputs(lengths, 1, K, K, seed=43, m_kind="householder", h_scale=0.1,
                                         init_scale=0.1)
    ref, rfin = oracle.cp_correct_varlen(H, M, h0, cu, "kv", "rev")
    fin = torch.empty((len(lengths), 1) + H.shape[2:], device="cuda:0")
    r = qla.cp_correct_varlen(_dev(H), _dev(M), _dev(cu.astype(np.int32)), _dev(h0), None, layout="kv",
                              direction="rev", final_state=fin, engine=engine, variant="scan", max_segments=30,
                              want_out=False)
    torch.cuda.synchronize()
    assert r is None and qla.device_status() == 0
    assert_parity(fin.cpu().numpy(), rfin, what=f"varlen scan final only {engine}")
    got, fin2 = _run(H, M, h0, cu, "kv", "rev", engine, variant="auto", max_segments=30)
    assert_parity(got, ref, what=f"varlen auto {engine}")
    assert_parity(fin2, rfin, what="varlen auto final")


@pytest.mark.parametrize("engine", engines_under_test())
def test_varlen_scan_bound_exceeded_is_flagged(engine):
    import torch

    import linear_attention_context_gb300 as qla
    K = 128
    if not engine_supports(engine, K, K):
        pytest.skip(f"engine {engine} does not take K={K}")
    H, M, h0, cu = qi.make_varlen_inputs([3, 9, 2], 2, K, K, seed=45)
    Hd, Md, h0d, cud = _dev(H), _dev(M), _dev(h0), _dev(cu.astype(np.int32))
    out = torch.zeros_like(Hd)
    qla.cp_correct_varlen(Hd, Md, cud, h0d, out, engine=engine, variant="scan", max_segments=4, scan_group=2)
    torch.cuda.synchronize()
    assert qla.device_status() == 2  # the 9-segment sequence exceeds the bound of 4
    # the sequences within the bound are still right
    ref, _ = oracle.cp_correct_varlen(H, M, h0, cu, "kv", "fwd")
    got = out.cpu().numpy()
    assert_parity(got[:, :3], ref[:, :3], what="first sequence next to an over-long one")
    assert_parity(got[:, 12:], ref[:, 12:], what="last sequence next to an over-long one")
    assert qla.device_status() == 0
