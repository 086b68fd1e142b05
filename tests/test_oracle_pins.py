"""Pins for the fp64 oracle: results fixed by mathematics, not by the oracle.

The pages print no values for the state correction, so the oracle is pinned by
(1) brute-force unrolled matrix products on tiny sizes, (2) closed forms for
M = I, M = 0, M = cI and the scalar K = V = 1 recurrence, (3) the layout and
direction identities, (4) exact integer cases, (5) norm invariants of the
orthogonal and Householder generators, and (6) a hand-derived 2x2 example.
test_oracle_mutants.py plants mistakes in a copy of the oracle and checks that
these pins catch them.
"""
import os

import numpy as np
import pytest

import oracle
import qla_inputs as qi
from qla_check import read_golden, to_kv, unrolled

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LAYOUTS = ("kv", "vk")
DIRS = ("fwd", "rev")


def rand_case(rng, B, nh, S, K, V, layout, with_init=True):
    st = (K, V) if layout == "kv" else (V, K)
    H = rng.standard_normal((B, nh, S) + st).astype(np.float32)
    M = (rng.standard_normal((B, nh, S, K, K)) / np.sqrt(K)).astype(np.float32)
    h0 = rng.standard_normal((B, nh) + st).astype(np.float32) if with_init else None
    return H, M, h0


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("K,V,S", [(1, 1, 1), (1, 1, 4), (2, 3, 3), (3, 2, 4), (8, 8, 4), (3, 5, 2)])
def test_unrolled_products(layout, direction, K, V, S):
    rng = np.random.default_rng(100 + K * 10 + V + S)
    H, M, h0 = rand_case(rng, 2, 2, S, K, V, layout)
    out, fin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
    uo, uf = unrolled(H, M, h0, layout, direction)
    np.testing.assert_allclose(out, uo, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin, uf, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("direction", DIRS)
def test_null_init_is_zero(layout, direction):
    rng = np.random.default_rng(7)
    H, M, _ = rand_case(rng, 1, 3, 4, 4, 6, layout, with_init=False)
    a, fa = oracle.cp_correct(H, M, None, layout, direction, want_final=True)
    z = np.zeros((1, 3) + H.shape[3:], np.float32)
    b, fb = oracle.cp_correct(H, M, z, layout, direction, want_final=True)
    assert np.array_equal(a, b) and np.array_equal(fa, fb)
    first = 0 if direction == "fwd" else H.shape[2] - 1
    assert not a[:, :, first].any()


@pytest.mark.parametrize("direction", DIRS)
def test_identity_is_prefix_sum(direction):
    c = qi.Case(B=1, heads=2, S=8, K=64, V=64, seed=11, m_kind="identity", h_kind="small_int",
                init_kind="small_int")
    H, M, h0 = qi.make_inputs(c)
    out, _ = oracle.cp_correct(H, M, h0, "kv", direction)
    H64 = H.astype(np.int64)
    for i in range(c.S):
        js = range(i) if direction == "fwd" else range(i + 1, c.S)
        exp = h0.astype(np.int64) + sum((H64[:, :, j] for j in js), np.zeros_like(h0, np.int64))
        assert np.array_equal(out[:, :, i], exp.astype(np.float64)), i


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("direction", DIRS)
def test_zero_M_passes_local_states(layout, direction):
    rng = np.random.default_rng(3)
    H, M, h0 = rand_case(rng, 1, 2, 5, 8, 4, layout)
    M[:] = 0
    out, _ = oracle.cp_correct(H, M, h0, layout, direction)
    S = H.shape[2]
    if direction == "fwd":
        assert np.array_equal(out[:, :, 0], h0.astype(np.float64))
        for i in range(1, S):
            assert np.array_equal(out[:, :, i], H[:, :, i - 1].astype(np.float64))
    else:
        assert np.array_equal(out[:, :, S - 1], h0.astype(np.float64))
        for i in range(S - 1):
            assert np.array_equal(out[:, :, i], H[:, :, i + 1].astype(np.float64))


@pytest.mark.parametrize("direction", DIRS)
def test_scalar_multiple_closed_form(direction):
    rng = np.random.default_rng(5)
    S, K, V, cc = 6, 4, 3, 0.5
    H, M, h0 = rand_case(rng, 1, 1, S, K, V, "kv")
    M[:] = cc * np.eye(K, dtype=np.float32)
    out, _ = oracle.cp_correct(H, M, h0, "kv", direction)
    Hd = H.astype(np.float64)
    for i in range(S):
        if direction == "fwd":
            exp = cc ** i * h0 + sum((cc ** (i - 1 - j) * Hd[:, :, j] for j in range(i)), 0.0)
        else:
            exp = cc ** (S - 1 - i) * h0 + sum((cc ** (j - 1 - i) * Hd[:, :, j] for j in range(i + 1, S)), 0.0)
        np.testing.assert_allclose(out[:, :, i], exp, rtol=1e-14, atol=1e-14)


def test_scalar_textbook_recurrence():
    # K = V = 1, m_i = 2, H_i = 1: x_{i+1} = 2 x_i + 1, so x_i = 2^i x_0 + 2^i - 1.
    S = 20
    H = np.ones((1, 1, S, 1, 1), np.float32)
    M = np.full((1, 1, S, 1, 1), 2.0, np.float32)
    h0 = np.full((1, 1, 1, 1), 3.0, np.float32)
    out, fin = oracle.cp_correct(H, M, h0, "kv", "fwd", want_final=True)
    for i in range(S):
        assert out[0, 0, i, 0, 0] == 2.0 ** i * 3 + 2.0 ** i - 1
    assert fin[0, 0, 0, 0] == 2.0 ** S * 3 + 2.0 ** S - 1


@pytest.mark.parametrize("direction", DIRS)
def test_layouts_are_transposes_bitwise(direction):
    rng = np.random.default_rng(9)
    H, M, h0 = rand_case(rng, 2, 2, 4, 16, 8, "kv")
    a, fa = oracle.cp_correct(H, M, h0, "kv", direction, want_final=True)
    Ht = np.ascontiguousarray(np.swapaxes(H, -1, -2))
    h0t = np.ascontiguousarray(np.swapaxes(h0, -1, -2))
    b, fb = oracle.cp_correct(Ht, M, h0t, "vk", direction, want_final=True)
    assert np.array_equal(a, np.swapaxes(b, -1, -2))
    assert np.array_equal(fa, np.swapaxes(fb, -1, -2))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_reverse_is_flipped_forward_bitwise(layout):
    rng = np.random.default_rng(13)
    H, M, h0 = rand_case(rng, 1, 3, 6, 8, 8, layout)
    r, rf = oracle.cp_correct(H, M, h0, layout, "rev", want_final=True)
    Hf = np.ascontiguousarray(H[:, :, ::-1])
    Mf = np.ascontiguousarray(np.swapaxes(M[:, :, ::-1], -1, -2))
    f, ff = oracle.cp_correct(Hf, Mf, h0, layout, "fwd", want_final=True)
    assert np.array_equal(r, f[:, :, ::-1])
    assert np.array_equal(rf, ff)


@pytest.mark.parametrize("direction", DIRS)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_integer_signed_permutation_exact(direction, layout):
    c = qi.Case(B=1, heads=2, S=8, K=32, V=16, seed=21, m_kind="signed_perm", h_kind="small_int",
                init_kind="small_int")
    H, M, h0 = qi.make_inputs(c, layout)
    out, _ = oracle.cp_correct(H, M, h0, layout, direction)
    # exact integer brute force
    Hk = to_kv(H, layout).astype(np.int64)
    Mi = M.astype(np.int64)
    x = to_kv(h0, layout).astype(np.int64)
    S = c.S
    order = range(S) if direction == "fwd" else range(S - 1, -1, -1)
    exp = np.zeros(Hk.shape, np.int64)
    for i in order:
        exp[:, :, i] = x
        A = Mi[:, :, i] if direction == "fwd" else np.swapaxes(Mi[:, :, i], -1, -2)
        x = np.einsum("bnkc,bncv->bnkv", A, x) + Hk[:, :, i]
    exp = exp if layout == "kv" else np.swapaxes(exp, -1, -2)
    assert np.array_equal(out, exp.astype(np.float64))
    assert np.abs(out).max() < 2 ** 24  # every value exact in fp32 as well


@pytest.mark.parametrize("direction", DIRS)
def test_orthogonal_scaled_norm(direction):
    c = qi.sweep_case(heads=2, S=8).with_(h_kind="zero")
    H, M, h0 = qi.make_inputs(c)
    # generator check: M / 0.99 is orthogonal to fp32 rounding
    Q = M.astype(np.float64) / 0.99
    err = np.abs(np.einsum("bnsij,bnsik->bnsjk", Q, Q) - np.eye(c.K)).max()
    assert err < 1e-5
    out, _ = oracle.cp_correct(H, M, h0, "kv", direction)
    n0 = np.sqrt((h0.astype(np.float64) ** 2).sum(axis=(-2, -1)))
    for j in range(c.S):
        i = j if direction == "fwd" else c.S - 1 - j
        ni = np.sqrt((out[:, :, i] ** 2).sum(axis=(-2, -1)))
        np.testing.assert_allclose(ni, 0.99 ** j * n0, rtol=1e-5)


def test_householder_norm_bound():
    c = qi.WORKLOADS["c0"].with_(init_kind="gaussian")
    H, M, h0 = qi.make_inputs(c)
    Md = M.astype(np.float64)
    # generator check: M = g (I - beta u u^T) is symmetric with spectral norm <= 1
    assert np.abs(Md - np.swapaxes(Md, -1, -2)).max() < 1e-6
    assert np.linalg.norm(Md.reshape(-1, c.K, c.K), ord=2, axis=(1, 2)).max() <= 1.0 + 1e-6
    out, fin = oracle.cp_correct(H, M, h0, "kv", "fwd", want_final=True)
    states = np.concatenate([out, fin[:, :, None]], axis=2)
    nrm = np.sqrt((states ** 2).sum(axis=(-2, -1)))
    nH = np.sqrt((H.astype(np.float64) ** 2).sum(axis=(-2, -1)))
    assert np.all(nrm[:, :, 1:] <= nrm[:, :, :-1] + nH + 1e-9)


def test_golden_hand_2x2():
    g = read_golden(os.path.join(GOLDEN, "hand_2x2_S3.txt"))
    H = np.stack([g["H0"], g["H1"], g["H2"]])[None, None].astype(np.float32)
    M = np.stack([g["M0"], g["M1"], g["M2"]])[None, None].astype(np.float32)
    h0 = g["h_init"][None, None].astype(np.float32)
    for d in DIRS:
        out, fin = oracle.cp_correct(H, M, h0, "kv", d, want_final=True)
        for i in range(3):
            assert np.array_equal(out[0, 0, i], g[f"{d}_out{i}"]), (d, i)
        assert np.array_equal(fin[0, 0], g[f"{d}_final"]), d


def test_thread_count_does_not_change_results():
    c = qi.WORKLOADS["c0"].with_(heads=4, init_kind="gaussian")
    H, M, h0 = qi.make_inputs(c, "vk")
    a, _, n1 = oracle.cp_correct(H, M, h0, "vk", "rev", nthreads=1, return_threads=True)
    b, _, n4 = oracle.cp_correct(H, M, h0, "vk", "rev", nthreads=4, return_threads=True)
    assert n1 == 1
    assert np.array_equal(a, b)
