"""Seeded random configurations against the fp64 oracle.

The state correction: shapes (K, V in 32 .. 256, S in 1 .. 40, B and heads),
M families, both layouts and directions, every engine that takes the shape,
both variants with random scan group counts, in place or not, a null h_init,
and the final state; long chains across the tensor-core engine's length
limit under the automatic choice; variable-length batches.  The local pass:
widths, segment counts and lengths, decay and write-strength ranges,
layouts, H or M alone, and sub-segment splits.  Each case comes from a fixed
seed, so a failure names a reproducible configuration; the bar is the parity
bar of the other tests.
"""
import numpy as np
import pytest

import oracle
import qla_inputs as qi
from gpu_util import engine_supports, run, run_varlen, to_dev
from qla_check import assert_parity

pytestmark = pytest.mark.gpu

WIDTHS = [32, 64, 96, 128, 160, 192, 224, 256]


def correction_case(i):
    r = np.random.default_rng(7000 + i)
    if r.random() < 0.5:  # half the cases in the tensor-core engine's widths
        K = int(r.choice([128, 256]))
    else:
        K = int(r.choice(WIDTHS))
    V = int(r.choice(WIDTHS))
    S = int(r.integers(1, 41))
    big = K >= 192 or V >= 192
    B = int(r.integers(1, 3))
    heads = int(r.integers(1, 2 if big else 4))
    m_kind = str(r.choice(["householder", "orthogonal", "signed_perm"]))
    init_kind = str(r.choice(["gaussian", "none"]))
    layout = str(r.choice(["kv", "vk"]))
    direction = str(r.choice(["fwd", "rev"]))
    engines = ["auto", "simt"] + (["tc"] if engine_supports("tc", K, V) else [])
    engine = str(r.choice(engines))
    variant = str(r.choice(["auto", "seq", "scan"]))
    group = int(r.integers(0, min(S, 12) + 1)) if variant == "scan" else 0
    in_place = bool(r.integers(0, 2))
    final = bool(r.integers(0, 2))
    case = qi.Case(B=B, heads=heads, S=S, K=K, V=V, seed=100 + i, m_kind=m_kind, h_scale=0.5,
                   init_kind=init_kind, init_scale=0.5)
    return case, layout, direction, engine, variant, group, in_place, final


@pytest.mark.parametrize("i", range(48))
def test_correction_random_configuration(i):
    c, layout, direction, engine, variant, group, in_place, final = correction_case(i)
    what = (f"case {i}: B={c.B} heads={c.heads} S={c.S} K={c.K} V={c.V} {c.m_kind} init={c.init_kind} "
            f"{layout}/{direction} engine={engine} variant={variant} group={group} in_place={in_place}")
    H, M, h0 = qi.make_inputs(c, layout)
    ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=final)
    out, fin = run(H, M, h0, layout, direction, engine=engine, variant=variant, in_place=in_place, final=final,
                   scan_group=group)
    assert_parity(out, ref, what=what)
    if final:
        assert_parity(fin, rfin, what=what + " final")


def local_case(i):
    r = np.random.default_rng(9000 + i)
    K = int(r.choice(WIDTHS))
    V = int(r.choice(WIDTHS))
    S = int(r.integers(1, 5))
    L = int(r.integers(1, 151))
    heads = int(r.integers(1, 3))
    alpha = [(0.9, 1.0), (0.999, 1.0), (0.6, 0.8), (0.5, 1.5)][int(r.integers(0, 4))]
    beta = [(0.0, 1.0), (0.0, 0.1), (0.5, 1.0)][int(r.integers(0, 3))]
    layout = str(r.choice(["kv", "vk"]))
    parts = [(True, True), (True, False), (False, True)][int(r.integers(0, 3))]
    splits = [0] + [f for f in (1, 2, 4, 8) if L % f == 0]
    split = int(r.choice(splits))
    case = qi.LocalCase(B=1, heads=heads, T=S * L, S=S, K=K, V=V, seed=300 + i, alpha_lo=alpha[0],
                        alpha_hi=alpha[1], beta_lo=beta[0], beta_hi=beta[1])
    return case, layout, parts, split


@pytest.mark.parametrize("i", range(32))
def test_local_pass_random_configuration(i):
    import torch
    import linear_attention_context_gb300 as qla
    c, layout, (want_H, want_M), split = local_case(i)
    what = (f"local case {i}: heads={c.heads} S={c.S} L={c.L} K={c.K} V={c.V} a=[{c.alpha_lo}, {c.alpha_hi}] "
            f"b=[{c.beta_lo}, {c.beta_hi}] {layout} H={want_H} M={want_M} split={split}")
    k, v, b, g = qi.make_local_inputs(c)
    Hr, Mr = oracle.local_pass(k, v, b, g, c.S, layout)
    H, M = qla.local_pass(*(to_dev(a) for a in (k, v, b, g)), c.S, layout=layout, want_H=want_H, want_M=want_M,
                          split=split)
    torch.cuda.synchronize()
    if want_H:
        assert_parity(H.cpu().numpy().astype(np.float64), Hr, what=what + " H")
    else:
        assert H is None
    if want_M:
        assert_parity(M.cpu().numpy().astype(np.float64), Mr, what=what + " M")
    else:
        assert M is None


@pytest.mark.parametrize("i", range(8))
def test_long_chain_random_configuration(i):
    """Chains of 40 to 200 segments (K <= 128) or 20 to 70 (K = 256) with the
    automatic engine, across the tensor-core engine's length limit, in either
    variant: the automatic choice must keep the bar."""
    r = np.random.default_rng(11000 + i)
    K = int(r.choice([64, 96, 128, 128, 256]))
    V = int(r.choice([32, 64, 128]))
    S = int(r.integers(40, 201)) if K <= 128 else int(r.integers(20, 71))
    heads = int(r.integers(1, 5))
    layout = str(r.choice(["kv", "vk"]))
    direction = str(r.choice(["fwd", "rev"]))
    variant = str(r.choice(["auto", "seq", "scan"]))
    c = qi.Case(B=1, heads=heads, S=S, K=K, V=V, seed=600 + i, m_kind=str(r.choice(["householder", "orthogonal"])),
                h_scale=0.3, init_scale=0.3)
    H, M, h0 = qi.make_inputs(c, layout)
    ref, rfin = oracle.cp_correct(H, M, h0, layout, direction, want_final=True)
    out, fin = run(H, M, h0, layout, direction, variant=variant, final=True)
    what = f"long case {i}: heads={heads} S={S} K={K} V={V} {c.m_kind} {layout}/{direction} {variant}"
    assert_parity(out, ref, what=what)
    assert_parity(fin, rfin, what=what + " final")


@pytest.mark.parametrize("i", range(16))
def test_varlen_random_configuration(i):
    """Variable-length batches: up to 8 sequences of 0 to 39 segments, every
    engine that takes the shape, both variants, with and without initial
    states."""
    r = np.random.default_rng(12000 + i)
    K = int(r.choice([64, 128, 256]))
    V = int(r.choice([32, 64, 128]))
    lengths = [int(x) for x in r.integers(0, 40, size=int(r.integers(1, 9)))]
    if sum(lengths) == 0:
        lengths[0] = 1
    heads = int(r.integers(1, 4))
    layout = str(r.choice(["kv", "vk"]))
    direction = str(r.choice(["fwd", "rev"]))
    engine = str(r.choice(["auto", "simt"] + (["tc"] if engine_supports("tc", K, V) else [])))
    variant = str(r.choice(["auto", "seq", "scan"]))
    with_init = bool(r.integers(0, 2))
    H, M, h0, cu = qi.make_varlen_inputs(lengths, heads, K, V, seed=800 + i, layout=layout, m_kind="orthogonal",
                                         h_scale=0.2, init_scale=0.2, with_init=with_init)
    ref, rfin = oracle.cp_correct_varlen(H, M, h0, cu, layout, direction)
    kw = {"variant": variant}
    if variant != "seq":
        kw["max_segments"] = max(lengths)
    got, fin = run_varlen(H, M, h0, cu, layout, direction, engine, **kw)
    what = f"varlen case {i}: {lengths} heads={heads} K={K} V={V} {layout}/{direction} {engine} {variant}"
    assert_parity(got, ref, what=what)
    assert_parity(fin, rfin, what=what + " final")
