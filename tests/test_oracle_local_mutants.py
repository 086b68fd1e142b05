"""Plants mistakes in a copy of the local-pass oracle (on the CPU) and checks
that the pins of test_oracle_local.py catch each one, and that the
chunked-form pin of test_oracle_local_chunked.py catches each one on its own:
the decay applied to the write term or left off the propagation matrix, a
write strength dropped from the removal term, the tokens visited backwards,
the propagation matrix started from zero, tokens shifted by one, the vk
layout left untransposed.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
import qla_inputs as qi
from oracle import build as obuild
from qla_check import local_products, read_golden

SRC = os.path.join(os.path.dirname(obuild.__file__), "qla_local_oracle.c")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "local_hand_2x2_L2.txt")

MUTANTS = {
    "decay_on_write": ("*x = at * (*x - bt * kt[a] * r[col]) + bt * kt[a] * vt[col];",
                       "*x = at * (*x - bt * kt[a] * r[col] + bt * kt[a] * vt[col]);"),
    "no_beta_in_removal": ("*x = at * (*x - bt * kt[a] * r[col]) + bt * kt[a] * vt[col];",
                           "*x = at * (*x - kt[a] * r[col]) + bt * kt[a] * vt[col];"),
    "no_decay_on_M": ("*p = at * (*p - bt * kt[a] * r[col]);", "*p = (*p - bt * kt[a] * r[col]);"),
    "tokens_backwards": ("for (int t = i * L; t < (i + 1) * L; ++t) {",
                         "for (int t = (i + 1) * L - 1; t >= i * L; --t) {"),
    "M_from_zero": ("P[(int64_t)a * K + b] = (a == b) ? 1.0 : 0.0;", "P[(int64_t)a * K + b] = 0.0;"),
    "tokens_shifted": ("const int64_t tok = c * T + t;", "const int64_t tok = c * T + (t + 1) % T;"),
    "vk_untransposed": ("h[layout == 0 ? (int64_t)a * V + col : (int64_t)col * K + a]", "h[(int64_t)a * V + col]"),
}


def build_mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    variant = f"_local_mutant_{name}"
    out_dir = os.path.dirname(obuild.library_path(variant))
    os.makedirs(out_dir, exist_ok=True)
    path = os.path.join(out_dir, f"local_mutant_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    cmd = obuild.build_command(variant=variant)
    cmd[cmd.index(SRC)] = path
    subprocess.run(cmd, check=True)
    return variant


def rand_tokens(rng, T, K, V):
    k = rng.standard_normal((1, 2, T, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, 2, T, V))
    b = rng.uniform(0, 1, size=(1, 2, T)).astype(np.float32)
    g = np.log(rng.uniform(0.7, 1, size=(1, 2, T))).astype(np.float32)
    return qi.f32_to_bf16(k.astype(np.float32)), qi.f32_to_bf16(v.astype(np.float32)), b, g


def pins_pass(variant):
    """A compact battery of the local-pass pins; False as soon as one fails."""
    rng = np.random.default_rng(7)
    for layout in ("kv", "vk"):
        for (K, V, T, S) in ((3, 4, 6, 2), (5, 5, 8, 4)):
            k, v, b, g = rand_tokens(rng, T, K, V)
            H, M = oracle.local_pass(k, v, b, g, S, layout, variant=variant)
            Hp, Mp = local_products(k, v, b, g, S, layout)
            if not (np.allclose(H, Hp, rtol=1e-12, atol=1e-13) and np.allclose(M, Mp, rtol=1e-12, atol=1e-13)):
                return False
    gd = read_golden(GOLDEN)
    k = qi.f32_to_bf16(np.stack([gd["k0"][0], gd["k1"][0]]).astype(np.float32))[None, None]
    v = qi.f32_to_bf16(np.stack([gd["v0"][0], gd["v1"][0]]).astype(np.float32))[None, None]
    b = np.array([[[gd["beta0"][0, 0], gd["beta1"][0, 0]]]], np.float32)
    g = np.array([[[gd["g0"][0, 0], gd["g1"][0, 0]]]], np.float32)
    H, M = oracle.local_pass(k, v, b, g, 1, variant=variant)
    return np.array_equal(H[0, 0, 0], gd["H"].reshape(2, 2)) and np.array_equal(M[0, 0, 0], gd["M"].reshape(2, 2))


def test_unmutated_local_oracle_passes_battery():
    assert pins_pass("")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_local_mutant(name):
    variant = build_mutant(name)
    assert not pins_pass(variant), f"mutant {name} slipped through the pins"


def chunked_pin_passes(variant):
    """The chunked-form pin alone (test_oracle_local_chunked.py): the oracle
    against a triangular solve per chunk, both layouts."""
    from test_oracle_local_chunked import chunked_local_pass
    rng = np.random.default_rng(11)
    for layout in ("kv", "vk"):
        k, v, b, g = rand_tokens(rng, 12, 4, 3)
        H, M = oracle.local_pass(k, v, b, g, 2, layout, variant=variant)
        Hc, Mc = chunked_local_pass(qi.bf16_to_f32(k).astype(np.float64), qi.bf16_to_f32(v).astype(np.float64),
                                    b, g, 2, 4)
        if layout == "vk":
            Hc = np.swapaxes(Hc, -1, -2)
        if not (np.allclose(H, Hc, rtol=1e-10, atol=1e-12) and np.allclose(M, Mc, rtol=1e-10, atol=1e-12)):
            return False
    return True


def test_unmutated_local_oracle_passes_chunked_pin():
    assert chunked_pin_passes("")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_chunked_pin_catches_local_mutant(name):
    variant = build_mutant(name)
    assert not chunked_pin_passes(variant), f"mutant {name} slipped through the chunked-form pin"
