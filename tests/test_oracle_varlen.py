"""Pins of the variable-length oracle (sequences of different segment counts
packed along the segment axis, offsets cu_seg).

Each (sequence, head) chain is the fixed-length recurrence over its own
segments.  The pins fix the packing from outside the oracle: with M = I the
outputs are per-sequence prefix sums (forward) or suffix sums (reverse), exact
for small integers; a one-segment sequence reduces to one explicit matrix
product; an empty sequence keeps its initial state; equal lengths reproduce the
fixed-length layout [N][heads][S] transposed to [heads][N*S].
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi

LENGTHS = [3, 0, 1, 5, 2, 0, 7]


def _int_inputs(lengths, heads, K, V, layout, seed):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    st = (K, V) if layout == "kv" else (V, K)
    H = rng.integers(-8, 9, (heads, T) + st).astype(np.float32)
    h0 = rng.integers(-8, 9, (len(lengths), heads) + st).astype(np.float32)
    M = np.broadcast_to(np.eye(K, dtype=np.float32), (heads, T, K, K)).copy()
    return H, M, h0, cu


@pytest.mark.parametrize("layout", ["kv", "vk"])
@pytest.mark.parametrize("direction", ["fwd", "rev"])
@pytest.mark.parametrize("with_init", [True, False])
def test_identity_gives_per_sequence_prefix_sums(layout, direction, with_init):
    H, M, h0, cu = _int_inputs(LENGTHS, 2, 4, 3, layout, seed=11)
    init = h0 if with_init else None
    out, fin = oracle.cp_correct_varlen(H, M, init, cu, layout, direction)
    for n in range(len(LENGTHS)):
        s0, s1 = cu[n], cu[n + 1]
        base = h0[n].astype(np.float64) if with_init else np.zeros(h0.shape[1:])
        for i in range(s0, s1):
            if direction == "fwd":
                want = base + H[:, s0:i].astype(np.float64).sum(axis=1)
            else:
                want = base + H[:, i + 1:s1].astype(np.float64).sum(axis=1)
            assert np.array_equal(out[:, i], want), (n, i)
        assert np.array_equal(fin[n], base + H[:, s0:s1].astype(np.float64).sum(axis=1)), n


@pytest.mark.parametrize("layout", ["kv", "vk"])
def test_one_segment_sequence_is_one_product(layout):
    H, M, h0, cu = qi.make_varlen_inputs([1, 2], 1, 6, 5, seed=3, layout=layout)
    out, fin = oracle.cp_correct_varlen(H, M, h0, cu, layout, "fwd")
    x0 = h0[0, 0].astype(np.float64)
    m0 = M[0, 0].astype(np.float64)
    assert np.array_equal(out[0, 0], x0)
    want = m0 @ x0 + H[0, 0] if layout == "kv" else x0 @ m0.T + H[0, 0]
    np.testing.assert_allclose(fin[0, 0], want, rtol=1e-14, atol=1e-14)


def test_empty_sequence_keeps_its_initial_state():
    H, M, h0, cu = qi.make_varlen_inputs([0, 3, 0], 2, 4, 4, seed=9)
    out, fin = oracle.cp_correct_varlen(H, M, h0, cu, "kv", "rev")
    assert np.array_equal(fin[0], h0[0]) and np.array_equal(fin[2], h0[2])
    out, fin = oracle.cp_correct_varlen(H, M, None, cu, "kv", "fwd")
    assert not fin[0].any() and not fin[2].any()


@pytest.mark.parametrize("layout,direction", [("kv", "fwd"), ("vk", "rev")])
def test_equal_lengths_match_fixed_layout(layout, direction):
    N, heads, S, K, V = 3, 2, 4, 8, 8
    c = qi.Case(B=N, heads=heads, S=S, K=K, V=V, seed=21)
    Hf, Mf, h0 = qi.make_inputs(c, layout)
    ref, rfin = oracle.cp_correct(Hf, Mf, h0, layout, direction, want_final=True)
    # [N][heads][S] -> [heads][N*S]
    H = np.ascontiguousarray(Hf.transpose((1, 0, 2) + tuple(range(3, Hf.ndim))).reshape((heads, N * S) + Hf.shape[3:]))
    M = np.ascontiguousarray(Mf.transpose(1, 0, 2, 3, 4).reshape(heads, N * S, K, K))
    cu = np.arange(0, N * S + 1, S, dtype=np.int32)
    out, fin = oracle.cp_correct_varlen(H, M, h0, cu, layout, direction)
    ref_packed = ref.transpose((1, 0, 2) + tuple(range(3, ref.ndim))).reshape(out.shape)
    assert np.array_equal(out, ref_packed)
    assert np.array_equal(fin, rfin)


def test_bad_offsets_are_rejected():
    H, M, h0, cu = qi.make_varlen_inputs([2, 2], 1, 4, 4, seed=1)
    for bad in ([0, 3, 2, 4], [1, 2, 4], [0, 2, 5]):
        with pytest.raises(AssertionError):
            oracle.cp_correct_varlen(H, M, None, np.array(bad), "kv", "fwd")
