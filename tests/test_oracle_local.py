"""Pins for the local-pass oracle (oracle.local_pass): values fixed by
mathematics, not by the oracle's own loop.

The oracle applies the gated delta rule token by token as rank-1 updates
(Gated Delta Networks, Yang, Kautz, Hatamizadeh, ICLR 2025, kv orientation):
X_t = a_t (I - b_t k_t k_t^T) X_{t-1} + b_t k_t v_t^T, a_t = exp(g_t); per
segment H = the state from zero, M = the product of the transitions.  Pins:
(1) explicit dense transition matrices multiplied in order (a product form
the oracle never builds); (2) orthogonal (basis) keys, where each token
overwrites one row: closed forms, bitwise on integers, with and without decay;
(3) no writes (b = 0): M = exp(sum g) I, H = 0; (4) composition of
sub-segments, the affine property the correction pass relies on; (5) the
correction oracle applied to the segments' (H, M) reproduces the whole
sequence's state at every segment boundary; (6) layouts are transposes;
(7) linearity in the values; (8) a hand-derived 2x2 example.
test_oracle_mutants.py plants mistakes in a copy of this oracle and checks
that these pins catch them.
"""
import os

import numpy as np
import pytest

import oracle
import qla_inputs as qi
from qla_check import local_products, read_golden

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_tokens(rng, B, nh, T, K, V, beta=(0.0, 1.0), alpha=(0.8, 1.0)):
    k = rng.standard_normal((B, nh, T, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, nh, T, V))
    b = rng.uniform(*beta, size=(B, nh, T)).astype(np.float32)
    g = np.log(rng.uniform(*alpha, size=(B, nh, T))).astype(np.float32)
    return qi.f32_to_bf16(k.astype(np.float32)), qi.f32_to_bf16(v.astype(np.float32)), b, g


@pytest.mark.parametrize("layout", ["kv", "vk"])
@pytest.mark.parametrize("K,V,T,S", [(1, 1, 3, 1), (2, 3, 4, 2), (3, 2, 6, 3), (5, 4, 6, 1), (4, 7, 8, 4),
                                     (8, 8, 12, 3)])
def test_explicit_matrix_products(layout, K, V, T, S):
    rng = np.random.default_rng(1000 + 97 * K + 13 * V + T + S)
    k, v, b, g = rand_tokens(rng, 2, 2, T, K, V)
    H, M = oracle.local_pass(k, v, b, g, S, layout)
    Hp, Mp = local_products(k, v, b, g, S, layout)
    np.testing.assert_allclose(M, Mp, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(H, Hp, rtol=1e-12, atol=1e-13)


def basis_case(K, V, T, S, seed, decay):
    """Keys are basis vectors e_j (exact in bf16), distinct inside a segment;
    values small integers; b = 1; decays a = 1 or 1/2."""
    rng = np.random.default_rng(seed)
    L = T // S
    idx = np.concatenate([rng.permutation(K)[:L] for _ in range(S)])
    kf = np.zeros((1, 1, T, K), np.float32)
    kf[0, 0, np.arange(T), idx] = 1.0
    vf = rng.integers(-8, 9, size=(1, 1, T, V)).astype(np.float32)
    b = np.ones((1, 1, T), np.float32)
    g = np.full((1, 1, T), np.float32(np.log(0.5)) if decay else 0.0, np.float32)
    return idx, qi.f32_to_bf16(kf), qi.f32_to_bf16(vf), vf, b, g


@pytest.mark.parametrize("decay", [False, True])
def test_orthogonal_keys_closed_form(decay):
    """With basis keys and b = 1 each token sets one row of the state to its
    value (the delta rule's write-then-read) and later tokens only decay it:
    H[j_t] = (product of the later decays) v_t, M = diag(decay product, or 0
    on the written rows)."""
    K, V, T, S = 16, 5, 12, 3
    L = T // S
    idx, k, v, vf, b, g = basis_case(K, V, T, S, 7, decay)
    H, M = oracle.local_pass(k, v, b, g, S, "kv")
    a = float(np.exp(np.float64(g[0, 0, 0])))
    for i in range(S):
        Hx = np.zeros((K, V))
        Mx = np.eye(K) * a ** L
        for j in range(L):
            t = i * L + j
            Hx[idx[t]] = a ** (L - 1 - j) * vf[0, 0, t].astype(np.float64)
            Mx[idx[t], idx[t]] = 0.0
        if decay:
            np.testing.assert_allclose(H[0, 0, i], Hx, rtol=1e-14, atol=0)
            np.testing.assert_allclose(M[0, 0, i], Mx, rtol=1e-14, atol=0)
        else:
            assert np.array_equal(H[0, 0, i], Hx)
            assert np.array_equal(M[0, 0, i], Mx)


def test_no_writes_leave_a_scaled_identity():
    rng = np.random.default_rng(3)
    k, v, _, g = rand_tokens(rng, 1, 3, 20, 6, 4, alpha=(0.5, 1.0))
    b = np.zeros((1, 3, 20), np.float32)
    H, M = oracle.local_pass(k, v, b, g, 4, "kv")
    assert np.array_equal(H, np.zeros_like(H))
    sums = g.astype(np.float64).reshape(1, 3, 4, 5).sum(-1)
    np.testing.assert_allclose(M, np.exp(sums)[..., None, None] * np.eye(6), rtol=1e-14, atol=0)


@pytest.mark.parametrize("layout", ["kv", "vk"])
def test_composition_of_sub_segments(layout):
    """Two halves composed as affine maps equal the whole segment:
    M = M_2 M_1, H = M_2 H_1 + H_2 (kv view)."""
    rng = np.random.default_rng(11)
    k, v, b, g = rand_tokens(rng, 1, 2, 24, 7, 5)
    Hw, Mw = oracle.local_pass(k, v, b, g, 1, "kv")
    Hh, Mh = oracle.local_pass(k, v, b, g, 2, "kv")
    np.testing.assert_allclose(Mw[:, :, 0], Mh[:, :, 1] @ Mh[:, :, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(Hw[:, :, 0], Mh[:, :, 1] @ Hh[:, :, 0] + Hh[:, :, 1], rtol=1e-12, atol=1e-14)
    if layout == "vk":
        Hv, _ = oracle.local_pass(k, v, b, g, 2, "vk")
        np.testing.assert_allclose(np.swapaxes(Hv, -1, -2), Hh, rtol=0, atol=0)


@pytest.mark.parametrize("layout", ["kv", "vk"])
def test_correction_of_segments_reproduces_the_whole_sequence(layout):
    """The correction oracle composing every segment's (H, M) from a zero
    start gives, at each segment boundary, the state of the whole sequence's
    token recurrence (the local pass over the tokens before that boundary)."""
    rng = np.random.default_rng(12)
    S, L = 5, 6
    k, v, b, g = rand_tokens(rng, 2, 2, S * L, 8, 6)
    H, M = oracle.local_pass(k, v, b, g, S, layout)
    out, fin = oracle.cp_correct(H.astype(np.float32), M.astype(np.float32), None, layout, "fwd",
                                 want_final=True)
    for i in range(1, S + 1):
        n = i * L
        Hp, _ = oracle.local_pass(k[:, :, :n], v[:, :, :n], b[:, :, :n], g[:, :, :n], 1, layout, want_M=False)
        got = fin if i == S else out[:, :, i]
        # the correction runs on fp32-rounded H and M: agree to fp32 rounding
        np.testing.assert_allclose(got, Hp[:, :, 0], rtol=2e-6, atol=2e-6 * np.abs(Hp).max())


def test_layouts_are_transposes_bitwise():
    rng = np.random.default_rng(13)
    k, v, b, g = rand_tokens(rng, 1, 2, 12, 5, 9)
    Hkv, Mkv = oracle.local_pass(k, v, b, g, 3, "kv")
    Hvk, Mvk = oracle.local_pass(k, v, b, g, 3, "vk")
    assert np.array_equal(np.swapaxes(Hvk, -1, -2), Hkv)
    assert np.array_equal(Mvk, Mkv)


def test_linear_in_the_values():
    """H is linear in v and M does not depend on v (exact on small integers)."""
    rng = np.random.default_rng(14)
    k, _, b, g = rand_tokens(rng, 1, 2, 9, 4, 3)
    v1 = rng.integers(-4, 5, size=(1, 2, 9, 3)).astype(np.float32)
    v2 = rng.integers(-4, 5, size=(1, 2, 9, 3)).astype(np.float32)
    H1, M1 = oracle.local_pass(k, qi.f32_to_bf16(v1), b, g, 3)
    H2, M2 = oracle.local_pass(k, qi.f32_to_bf16(v2), b, g, 3)
    H3, M3 = oracle.local_pass(k, qi.f32_to_bf16(v1 + 3 * v2), b, g, 3)
    assert np.array_equal(M1, M2) and np.array_equal(M1, M3)
    np.testing.assert_allclose(H3, H1 + 3 * H2, rtol=1e-13, atol=1e-13 * np.abs(H3).max())


def test_hand_derived_example():
    gd = read_golden(os.path.join(GOLDEN, "local_hand_2x2_L2.txt"))
    k = qi.f32_to_bf16(np.stack([gd["k0"][0], gd["k1"][0]]).astype(np.float32))[None, None]
    v = qi.f32_to_bf16(np.stack([gd["v0"][0], gd["v1"][0]]).astype(np.float32))[None, None]
    b = np.array([[[gd["beta0"][0, 0], gd["beta1"][0, 0]]]], np.float32)
    g = np.array([[[gd["g0"][0, 0], gd["g1"][0, 0]]]], np.float32)
    H, M = oracle.local_pass(k, v, b, g, 1)
    assert np.array_equal(H[0, 0, 0], gd["H"].reshape(2, 2))
    assert np.array_equal(M[0, 0, 0], gd["M"].reshape(2, 2))
    H2, M2 = oracle.local_pass(k, v, b, g, 2)
    for i in range(2):
        assert np.array_equal(H2[0, 0, i], gd[f"H_seg{i}"].reshape(2, 2))
        assert np.array_equal(M2[0, 0, i], gd[f"M_seg{i}"].reshape(2, 2))


def test_thread_count_does_not_change_results():
    c = qi.LOCAL_WORKLOADS["l0"].with_(heads=3)
    k, v, b, g = qi.make_local_inputs(c)
    H1, M1 = oracle.local_pass(k, v, b, g, c.S, nthreads=1)
    H4, M4 = oracle.local_pass(k, v, b, g, c.S, nthreads=4)
    assert np.array_equal(H1, H4) and np.array_equal(M1, M4)


def test_generated_workload_is_well_scaled():
    """The input recipe: unit keys (to bf16 rounding), write strengths and
    decays in their ranges, and segment propagation matrices far from zero
    and inside fp32's range."""
    c = qi.LOCAL_WORKLOADS["l0"]
    k, v, b, g = qi.make_local_inputs(c)
    kn = np.linalg.norm(qi.bf16_to_f32(k).astype(np.float64), axis=-1)
    assert np.all(np.abs(kn - 1) < 1e-2)
    assert b.min() >= c.beta_lo and b.max() < c.beta_hi
    assert g.max() <= 0 and g.min() >= np.log(c.alpha_lo) - 1e-6
    _, M = oracle.local_pass(k, v, b, g, c.S)
    fro = np.linalg.norm(M, axis=(-2, -1))
    assert np.all(fro > 1e-3) and np.all(fro < 10)
