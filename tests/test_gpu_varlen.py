"""GPU parity of the variable-length form (qla_cp_correct_varlen) against the
fp64 varlen oracle: sequences of different segment counts, including empty
and one-segment sequences, both layouts and directions, both engines, with
and without initial states, in place; and the device-side check of the
offsets (a chain with invalid offsets is skipped and flagged).
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi
from gpu_util import engine_supports, engines_under_test
from qla_check import assert_parity

pytestmark = pytest.mark.gpu

LENGTHS = [3, 0, 1, 8, 2, 0, 5, 13]


def _dev(a):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


def _run(H, M, h0, cu, layout, direction, engine, in_place=False):
    import torch

    import linear_attention_context_gb300 as qla
    Hd, Md, h0d = _dev(H), _dev(M), _dev(h0)
    cud = _dev(cu.astype(np.int32))
    N, heads = len(cu) - 1, H.shape[0]
    fin = torch.empty((N, heads) + H.shape[2:], device="cuda:0")
    out = Hd if in_place else None
    out = qla.cp_correct_varlen(Hd, Md, cud, h0d, out, layout=layout, direction=direction, final_state=fin,
                                engine=engine)
    torch.cuda.synchronize()
    assert qla.device_status() == 0
    return out.cpu().numpy(), fin.cpu().numpy()


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
