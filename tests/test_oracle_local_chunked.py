"""A pin for the local-pass oracle from a second formulation: the chunked form
of the gated delta rule.

The oracle applies the rule token by token as rank-1 updates.  The chunked
form (the one "Gated Delta Networks", Yang, Kautz, Hatamizadeh, ICLR 2025,
computes on tensor cores) reaches the same states through a triangular
solve per chunk of C tokens instead.  With the rule written as
X_t = a_t X_{t-1} + k_t u_t^T and u_t = b_t (v_t - a_t X_{t-1}^T k_t), the
chunk's cumulative decays g_t = a_1 ... a_t give

    (I + A) U = diag(b) V - diag(b g) K X_0,
    A[t, s] = b_t (g_t / g_s) (k_t . k_s)  for s < t, else 0,
    X_C = g_C X_0 + Khat^T U,   Khat_t = (g_C / g_t) k_t,

so H (from X_0 = 0) and M (from X_0 = I with V = 0) follow chunk by chunk.
This is fp64 numpy with a library solve, written from the derivation above;
it shares nothing with the oracle's loop.  The two must agree to rounding
for every chunk size, including one chunk per token (C = 1) and one chunk
per segment (C = L).
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi


def chunked_local_pass(kf, vf, b, g, S, C):
    """H [..., S, K, V] and M [..., S, K, K] in the kv view, fp64, by chunks of C tokens."""
    B, nh, T, K = kf.shape
    V = vf.shape[-1]
    L = T // S
    H = np.zeros((B, nh, S, K, V))
    M = np.zeros((B, nh, S, K, K))
    for bb in range(B):
        for h in range(nh):
            for s in range(S):
                XH = np.zeros((K, V))
                XM = np.eye(K)
                for c0 in range(s * L, (s + 1) * L, C):
                    c1 = min(c0 + C, (s + 1) * L)
                    k = kf[bb, h, c0:c1]            # [n, K]
                    v = vf[bb, h, c0:c1]            # [n, V]
                    bt = b[bb, h, c0:c1].astype(np.float64)
                    gc = np.cumsum(g[bb, h, c0:c1].astype(np.float64))  # log g_t
                    ratio = np.exp(gc[:, None] - gc[None, :])          # g_t / g_s
                    A = np.tril(bt[:, None] * ratio * (k @ k.T), -1)
                    T_ = np.eye(len(bt)) + A
                    bg = bt * np.exp(gc)
                    khat = np.exp(gc[-1] - gc)[:, None] * k
                    UH = np.linalg.solve(T_, bt[:, None] * v - bg[:, None] * (k @ XH))
                    XH = np.exp(gc[-1]) * XH + khat.T @ UH
                    UM = np.linalg.solve(T_, -bg[:, None] * (k @ XM))
                    XM = np.exp(gc[-1]) * XM + khat.T @ UM
                H[bb, h, s] = XH
                M[bb, h, s] = XM
    return H, M


def tokens(seed, B, nh, T, K, V, beta, alpha):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((B, nh, T, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, nh, T, V))
    b = rng.uniform(*beta, size=(B, nh, T)).astype(np.float32)
    g = np.log(rng.uniform(*alpha, size=(B, nh, T))).astype(np.float32)
    kb, vb = qi.f32_to_bf16(k.astype(np.float32)), qi.f32_to_bf16(v.astype(np.float32))
    return kb, vb, b, g


@pytest.mark.parametrize("C", [1, 3, 8, 24])
@pytest.mark.parametrize("alpha,beta", [((0.7, 1.0), (0.0, 1.0)), ((0.95, 1.0), (0.5, 1.0)),
                                        ((0.5, 1.5), (0.0, 0.5))])
def test_chunked_form_matches_the_token_recurrence(C, alpha, beta):
    B, nh, S, L, K, V = 1, 2, 2, 24, 8, 5
    kb, vb, b, g = tokens(C * 7 + int(alpha[0] * 100), B, nh, S * L, K, V, beta, alpha)
    Hr, Mr = oracle.local_pass(kb, vb, b, g, S, "kv")
    kf = qi.bf16_to_f32(kb).astype(np.float64)
    vf = qi.bf16_to_f32(vb).astype(np.float64)
    Hc, Mc = chunked_local_pass(kf, vf, b, g, S, C)
    np.testing.assert_allclose(Hc, Hr, rtol=0, atol=1e-11 * np.abs(Hr).max())
    np.testing.assert_allclose(Mc, Mr, rtol=0, atol=1e-11 * np.abs(Mr).max())


def test_chunked_form_in_the_vk_layout():
    B, nh, S, L, K, V = 1, 1, 3, 10, 6, 7
    kb, vb, b, g = tokens(5, B, nh, S * L, K, V, (0.0, 1.0), (0.8, 1.0))
    Hr, Mr = oracle.local_pass(kb, vb, b, g, S, "vk")
    Hc, Mc = chunked_local_pass(qi.bf16_to_f32(kb).astype(np.float64), qi.bf16_to_f32(vb).astype(np.float64),
                                b, g, S, 4)
    np.testing.assert_allclose(np.swapaxes(Hc, -1, -2), Hr, rtol=0, atol=1e-11 * np.abs(Hr).max())
    np.testing.assert_allclose(Mc, Mr, rtol=0, atol=1e-11 * np.abs(Mr).max())
