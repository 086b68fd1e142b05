"""Shared checks for the tests: the parity tolerance, an unrolled brute-force
form of the recurrence, and the slot-generation forensics.

Nothing here is imported by the library.
"""
from __future__ import annotations

import numpy as np

# Parity bar per output state (b, h, i): relative L2 error and max error
# relative to the state's largest magnitude.  A state whose reference is all
# zero must match exactly.
REL_L2 = 1e-5
REL_MAX = 1e-4


def state_errors(got, ref):
    """Per-state (rel-L2, max-abs / max|ref|) over the last two axes."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    lead = got.shape[:-2]
    # one row per state, so every reduction runs along contiguous memory
    g = got.reshape(-1, got.shape[-2] * got.shape[-1])
    r = ref.reshape(g.shape)
    d = g - r
    num = np.sqrt(np.einsum("ij,ij->i", d, d)).reshape(lead)
    den = np.sqrt(np.einsum("ij,ij->i", r, r)).reshape(lead)
    # max |x| as max(max x, -min x): no second large temporary
    mref = np.maximum(r.max(axis=1), -r.min(axis=1)).reshape(lead)
    mabs = np.maximum(d.max(axis=1), -d.min(axis=1)).reshape(lead)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(den > 0, num / np.where(den > 0, den, 1), np.where(num > 0, np.inf, 0.0))
        rmax = np.where(mref > 0, mabs / np.where(mref > 0, mref, 1), np.where(mabs > 0, np.inf, 0.0))
    return rel, rmax


def assert_parity(got, ref, rel_l2=REL_L2, rel_max=REL_MAX, what=""):
    rel, rmax = state_errors(got, ref)
    bad = (rel > rel_l2) | (rmax > rel_max) | ~np.isfinite(rel) | ~np.isfinite(rmax)
    if bad.any():
        idx = np.argwhere(bad)
        worst = np.unravel_index(np.nanargmax(np.where(np.isfinite(rel), rel, 1e300)), rel.shape)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} states out of tolerance; first {idx[:5].tolist()}; "
            f"worst rel-L2 {rel[worst]:.3e} at {worst}, max rel-max {np.nanmax(rmax):.3e}")
    return float(np.max(rel)) if rel.size else 0.0, float(np.max(rmax)) if rmax.size else 0.0


def to_kv(x, layout):
    """kv view (... K, V) of a state array stored in ``layout``."""
    return x if layout == "kv" else np.swapaxes(x, -1, -2)


def unrolled(H, M, h_init, layout, direction):
    """Brute force: every output written as a sum of explicit matrix products.

    forward: out[i] = (M_{i-1} ... M_0) h + sum_{j<i} (M_{i-1} ... M_{j+1}) H_j
    reverse: out[i] = (M_{i+1}^T ... M_{S-1}^T) h + sum_{j>i} (M_{i+1}^T ... M_{j-1}^T) H_j
    final:   the same with i = S (forward) or i = -1 (reverse).
    Returns (out, final) in ``layout``, fp64."""
    Hk = to_kv(np.asarray(H, np.float64), layout)
    M = np.asarray(M, np.float64)
    B, nh, S, K, V = Hk.shape
    h = np.zeros((B, nh, K, V)) if h_init is None else to_kv(np.asarray(h_init, np.float64), layout)
    out = np.zeros((B, nh, S + 1, K, V))  # slot S holds the final state

    def prod(b, n, lo, hi, transpose):
        # forward: M_{hi} ... M_{lo}; reverse: M_{lo}^T ... M_{hi}^T (identity if hi < lo)
        P = np.eye(K)
        for t in range(lo, hi + 1):
            m = M[b, n, t]
            P = (m @ P) if not transpose else (P @ m.T)
        return P

    for b in range(B):
        for n in range(nh):
            for i in range(S + 1):
                if direction == "fwd":
                    acc = prod(b, n, 0, i - 1, False) @ h[b, n]
                    for j in range(i):
                        acc = acc + prod(b, n, j + 1, i - 1, False) @ Hk[b, n, j]
                else:
                    ii = i if i < S else -1  # slot S holds the reverse final state (i = -1)
                    acc = prod(b, n, ii + 1, S - 1, True) @ h[b, n]
                    for j in range(ii + 1, S):
                        acc = acc + prod(b, n, ii + 1, j - 1, True) @ Hk[b, n, j]
                out[b, n, i] = acc
    o = out[:, :, :S]
    f = out[:, :, S]
    if layout == "vk":
        o = np.swapaxes(o, -1, -2)
        f = np.swapaxes(f, -1, -2)
    return o, f


def generation_forensics(got, ref, H, direction):
    """Slot-generation forensics for exact (integer) cases.

    For the elements of the first wrong output state (in processing order),
    takes the local-state term the kernel actually added,
    ``got - (ref - H[src])``, and counts how often it equals, at the same
    coordinates, the H of the segment two steps later or earlier: the
    double-buffer slot's next or previous generation.  ``src`` is the segment
    whose H built that output (i-1 forward, i+1 reverse).  With M = 0 the term
    is simply ``got``.  Returns a dict of counts."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    H = np.asarray(H, np.float64)
    S = got.shape[2]
    res = {"mismatch": int((got != ref).sum()), "first_state": None, "first_state_wrong": 0,
           "equals_H_plus2": 0, "equals_H_minus2": 0}
    order = range(S) if direction == "fwd" else range(S - 1, -1, -1)
    for i in order:
        w = got[:, :, i] != ref[:, :, i]
        if not w.any():
            continue
        src = i - 1 if direction == "fwd" else i + 1
        res["first_state"] = i
        res["first_state_wrong"] = int(w.sum())
        if 0 <= src < S:
            added = got[:, :, i] - (ref[:, :, i] - H[:, :, src])
            for shift, key in ((2, "equals_H_plus2"), (-2, "equals_H_minus2")):
                k = src + shift
                if 0 <= k < S:
                    res[key] = int((w & (added == H[:, :, k])).sum())
        break
    return res


def read_golden(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, rhs = (s.strip() for s in line.split("=", 1))
            rows = [[float(x) for x in r.split()] for r in rhs.split(";")]
            vals[name] = np.array(rows, np.float64)
    return vals


def bf16_bits_to_f64(a):
    """Exact values of bf16 bit patterns (int16 or uint16 arrays)."""
    return (np.asarray(a).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def local_products(k, v, beta, g, S, layout="kv"):
    """Brute force for the local pass: every token's transition formed as a
    dense matrix, A_t = a_t (I - b_t k_t k_t^T) with a_t = exp(g_t), and per
    segment M = A_last ... A_first, H = sum_t (A_last ... A_{t+1}) b_t k_t v_t^T
    (kv view; transposed for vk).  Returns (H, M) in fp64."""
    kf = bf16_bits_to_f64(k)
    vf = bf16_bits_to_f64(v)
    B, nh, T, K = kf.shape
    V = vf.shape[-1]
    L = T // S
    H = np.zeros((B, nh, S, K, V))
    M = np.zeros((B, nh, S, K, K))
    for b in range(B):
        for n in range(nh):
            for i in range(S):
                seg = range(i * L, (i + 1) * L)
                A = [np.exp(np.float64(g[b, n, t])) * (np.eye(K) - np.float64(beta[b, n, t]) *
                                                        np.outer(kf[b, n, t], kf[b, n, t])) for t in seg]
                Mi = np.eye(K)
                for At in A:
                    Mi = At @ Mi
                Hi = np.zeros((K, V))
                for j, t in enumerate(seg):
                    P = np.eye(K)
                    for At in A[j + 1:]:
                        P = At @ P
                    Hi += P @ (np.float64(beta[b, n, t]) * np.outer(kf[b, n, t], vf[b, n, t]))
                M[b, n, i] = Mi
                H[b, n, i] = Hi
    if layout == "vk":
        H = np.swapaxes(H, -1, -2)
    return H, M
