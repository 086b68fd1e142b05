"""Plants mistakes in a copy of the oracle (on the CPU) and checks that the pins
catch each one: a transposed operand, a dropped or negated term, a wrong
segment or output index, a wrong traversal order, a wrong vk index.  The last
mutant reads the local state of the segment two steps ahead, as a reused
double-buffer slot would, and checks that the slot-generation forensics used by
the GPU race tests name it.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import build as obuild
from qla_check import generation_forensics, read_golden, unrolled

SRC = os.path.join(os.path.dirname(obuild.__file__), "qla_oracle.c")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_2x2_S3.txt")

MUTANTS = {
    "transposed_M": ("reverse ? (double)Mseg[(int64_t)c * K + k] : (double)Mseg[(int64_t)k * K + c]",
                     "reverse ? (double)Mseg[(int64_t)k * K + c] : (double)Mseg[(int64_t)c * K + k]"),
    "dropped_H": ("if (Hseg) acc += ", "if (0) acc += "),
    "negated_H": ("if (Hseg) acc += ", "if (Hseg) acc -= "),
    "shifted_output": ("double* o = out + (c * S + i) * st;",
                       "double* o = out + (c * S + (direction == 0 ? (i + 1) % S : (i + S - 1) % S)) * st;"),
    "wrong_M_segment": ("step(Mc + (int64_t)i * K * K,", "step(Mc + (int64_t)(S - 1 - i) * K * K,"),
    "vk_as_kv": ("return layout == 0 ? (int64_t)k * V + v : (int64_t)v * K + k;",
                 "return (int64_t)k * V + v;"),
    "no_reverse_order": ("const int i = direction == 0 ? j : S - 1 - j;", "const int i = j;"),
    "next_generation_H": ("Hc + (int64_t)i * st,", "Hc + (int64_t)(i + 2 < S ? i + 2 : i) * st,"),
}


def build_mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    variant = f"_mutant_{name}"
    out_dir = os.path.dirname(obuild.library_path(variant))
    os.makedirs(out_dir, exist_ok=True)
    path = os.path.join(out_dir, f"mutant_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    cmd = obuild.build_command(variant=variant)
    cmd[cmd.index(SRC)] = path
    subprocess.run(cmd, check=True)
    return variant


def pins_pass(variant):
    """A compact battery of the pins; False as soon as one fails."""
    rng = np.random.default_rng(42)
    for layout in ("kv", "vk"):
        for d in ("fwd", "rev"):
            for (K, V, S) in ((3, 5, 3), (2, 2, 4)):
                st = (K, V) if layout == "kv" else (V, K)
                H = rng.standard_normal((1, 2, S) + st).astype(np.float32)
                M = rng.standard_normal((1, 2, S, K, K)).astype(np.float32)
                h0 = rng.standard_normal((1, 2) + st).astype(np.float32)
                out, fin = oracle.cp_correct(H, M, h0, layout, d, want_final=True, variant=variant)
                uo, uf = unrolled(H, M, h0, layout, d)
                if not (np.allclose(out, uo, rtol=1e-12, atol=1e-12)
                        and np.allclose(fin, uf, rtol=1e-12, atol=1e-12)):
                    return False
    g = read_golden(GOLDEN)
    H = np.stack([g["H0"], g["H1"], g["H2"]])[None, None].astype(np.float32)
    M = np.stack([g["M0"], g["M1"], g["M2"]])[None, None].astype(np.float32)
    h0 = g["h_init"][None, None].astype(np.float32)
    for d in ("fwd", "rev"):
        out, fin = oracle.cp_correct(H, M, h0, "kv", d, want_final=True, variant=variant)
        for i in range(3):
            if not np.array_equal(out[0, 0, i], g[f"{d}_out{i}"]):
                return False
        if not np.array_equal(fin[0, 0], g[f"{d}_final"]):
            return False
    return True


def test_unmutated_oracle_passes_battery():
    assert pins_pass("")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    variant = build_mutant(name)
    assert not pins_pass(variant), f"mutant {name} slipped through the pins"


@pytest.mark.parametrize("direction", ["fwd"])
def test_forensics_names_next_generation(direction):
    """With M = 0 (no propagation, as in the page's isolation step), the planted
    slot-reuse mutant's wrong values equal H two segments ahead."""
    variant = build_mutant("next_generation_H")
    rng = np.random.default_rng(1)
    S, K, V = 8, 8, 8
    H = rng.integers(-8, 9, (1, 2, S, K, V)).astype(np.float32)
    M = np.zeros((1, 2, S, K, K), np.float32)
    h0 = rng.integers(-8, 9, (1, 2, K, V)).astype(np.float32)
    good, _ = oracle.cp_correct(H, M, h0, "kv", direction)
    bad, _ = oracle.cp_correct(H, M, h0, "kv", direction, variant=variant)
    rep = generation_forensics(bad, good, H, direction)
    assert rep["first_state"] == 1
    assert rep["equals_H_plus2"] == rep["first_state_wrong"] > 0
    rep0 = generation_forensics(good, good, H, direction)
    assert rep0["mismatch"] == 0 and rep0["first_state"] is None
