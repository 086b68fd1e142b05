"""Randomised properties of the oracle over small random shapes (hypothesis).

Each property holds exactly for the recurrence, whatever the shapes:
- the oracle equals the brute-force unrolled products (fp64 rounding aside);
- kv and vk results are transposes of each other (bitwise);
- reverse equals forward on reversed segments with transposed M (bitwise);
- the map (H, h_init) -> outputs is linear.
The fixed-case pins cover named closed forms; these cover the shape space.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from qla_check import unrolled  # noqa: E402

shapes = st.tuples(st.integers(1, 2), st.integers(1, 2), st.integers(1, 5), st.integers(1, 6), st.integers(1, 6))


def _inputs(shape, seed, layout, with_init=True):
    B, nh, S, K, V = shape
    rng = np.random.default_rng(seed)
    st_ = (K, V) if layout == "kv" else (V, K)
    H = rng.standard_normal((B, nh, S) + st_).astype(np.float32)
    M = (rng.standard_normal((B, nh, S, K, K)) / np.sqrt(K)).astype(np.float32)
    h0 = rng.standard_normal((B, nh) + st_).astype(np.float32) if with_init else None
    return H, M, h0


@settings(max_examples=60, deadline=None)
@given(shape=shapes, seed=st.integers(0, 2**31 - 1), layout=st.sampled_from(["kv", "vk"]),
       direction=st.sampled_from(["fwd", "rev"]), with_init=st.booleans())
def test_matches_unrolled_products(shape, seed, layout, direction, with_init):
    H, M, h0 = _inputs(shape, seed, layout, with_init)
    out, fin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
    uo, uf = unrolled(H, M, h0, layout, direction)
    np.testing.assert_allclose(out, uo, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(fin, uf, rtol=1e-11, atol=1e-11)


@settings(max_examples=60, deadline=None)
@given(shape=shapes, seed=st.integers(0, 2**31 - 1), direction=st.sampled_from(["fwd", "rev"]))
def test_kv_vk_transpose(shape, seed, direction):
    H, M, h0 = _inputs(shape, seed, "kv")
    kv, kf = oracle.cp_correct(H, M, h0, "kv", direction, want_final=True)
    vk, vf = oracle.cp_correct(np.swapaxes(H, -1, -2), M, np.swapaxes(h0, -1, -2), "vk", direction, want_final=True)
    assert np.array_equal(kv, np.swapaxes(vk, -1, -2))
    assert np.array_equal(kf, np.swapaxes(vf, -1, -2))


@settings(max_examples=60, deadline=None)
@given(shape=shapes, seed=st.integers(0, 2**31 - 1), layout=st.sampled_from(["kv", "vk"]))
def test_reverse_is_flipped_forward(shape, seed, layout):
    H, M, h0 = _inputs(shape, seed, layout)
    rev, rf = oracle.cp_correct(H, M, h0, layout, "rev", want_final=True)
    fwd, ff = oracle.cp_correct(H[:, :, ::-1], np.swapaxes(M[:, :, ::-1], -1, -2), h0, layout, "fwd",
                                want_final=True)
    assert np.array_equal(rev, fwd[:, :, ::-1])
    assert np.array_equal(rf, ff)


@settings(max_examples=40, deadline=None)
@given(shape=shapes, seed=st.integers(0, 2**31 - 1), layout=st.sampled_from(["kv", "vk"]),
       direction=st.sampled_from(["fwd", "rev"]))
def test_linear_in_states(shape, seed, layout, direction):
    H1, M, h1 = _inputs(shape, seed, layout)
    H2, _, h2 = _inputs(shape, seed + 1, layout)
    a, af = oracle.cp_correct(H1, M, h1, layout, direction, want_final=True)
    b, bf = oracle.cp_correct(H2, M, h2, layout, direction, want_final=True)
    # the sums are exact in fp64 only up to rounding of the fp32 inputs' sum: use fp64 inputs' sum
    Hs = (H1.astype(np.float64) + H2).astype(np.float32)
    hs = (h1.astype(np.float64) + h2).astype(np.float32)
    c, cf = oracle.cp_correct(Hs, M, hs, layout, direction, want_final=True)
    dH = Hs.astype(np.float64) - H1 - H2  # rounding of the fp32 sum, propagated linearly
    dh = hs.astype(np.float64) - h1 - h2
    d, df = oracle.cp_correct(dH, M, dh, layout, direction, want_final=True) if (dH.any() or dh.any()) else (0, 0)
    scale = max(1.0, np.abs(c).max(), np.abs(cf).max())
    np.testing.assert_allclose(c, a + b + d, rtol=0, atol=1e-10 * scale)
    np.testing.assert_allclose(cf, af + bf + df, rtol=0, atol=1e-10 * scale)
