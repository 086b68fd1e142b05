"""Slot-reuse race replay on the warp-specialised engine.

The page this pass comes from (Antarx Memos, "一次 TileLang Warp Specialization
数值错误的定位与修复") found a double-buffer slot released before its last
ordinary read: the wrong values were, element for element, the local state of
the segment two steps later (forward) or earlier (reverse) -- the slot's next
generation.  It also found that isolated replays could hide the race and
that only replays at the real call site, repeated and with the same
arguments, exposed it (sections "第一个弯路" and "决定性证据").  These tests
replay the pipeline the same way:

- in place (out == H) and into separate outputs,
- many calls back to back on one stream with no synchronisation,
- two input sets alternating, with and without an L2-thrashing write between
  calls,
- on exact-integer inputs (signed-permutation M, small-integer states), so
  every correct result is bitwise equal to the oracle, and any mismatch is
  checked against the neighbouring generations of H.
"""
import numpy as np
import pytest

import linear_attention_context_gb300 as qla
import oracle
import qla_inputs as qi
from gpu_util import engine_supports, engines_under_test
from qla_check import generation_forensics

pytestmark = pytest.mark.gpu

REPS = 50
CASES = (("vk", "fwd"), ("kv", "rev"), ("kv", "fwd"), ("vk", "rev"))


def exact_case(seed):
    return qi.Case(B=1, heads=32, S=8, K=128, V=128, seed=seed, m_kind="signed_perm", h_kind="small_int",
                   init_kind="small_int")


def prepare(layout, direction, seeds=(31, 32)):
    import torch
    dev = torch.device("cuda:0")
    sets = []
    for sd in seeds:
        H, M, h0 = qi.make_inputs(exact_case(sd), layout)
        ref, _ = oracle.cp_correct(H, M, h0, layout, direction)
        sets.append(dict(H=H, ref=ref, Hd=torch.from_numpy(H).to(dev), Md=torch.from_numpy(M).to(dev),
                         h0d=torch.from_numpy(h0).to(dev)))
    return sets


def check_all(results, sets, direction, what):
    for it, out in enumerate(results):
        s = sets[it % len(sets)]
        got = out.cpu().numpy().astype(np.float64)
        if not np.array_equal(got, s["ref"]):
            rep = generation_forensics(got, s["ref"], s["H"], direction)
            raise AssertionError(f"{what}: call {it} differs from the oracle; forensics {rep}")


@pytest.mark.parametrize("release", ["membar", "proxy", "delay"])
@pytest.mark.parametrize("thrash", [False, True])
@pytest.mark.parametrize("layout,direction", CASES)
@pytest.mark.parametrize("engine", [e for e in engines_under_test() if e != "simt"] or ["simt"])
def test_back_to_back_replay(engine, layout, direction, thrash, release):
    import torch
    if not engine_supports(engine, 128, 128):
        pytest.skip("shape")
    sets = prepare(layout, direction)
    scratch = torch.empty(64 << 20, dtype=torch.float32, device="cuda:0") if thrash else None  # 256 MB
    results = []
    for it in range(REPS):
        s = sets[it % 2]
        out = torch.empty_like(s["Hd"])
        qla.cp_correct(s["Hd"], s["Md"], s["h0d"], out, layout=layout, direction=direction, engine=engine,
                       release=release)
        results.append(out)
        if thrash:
            scratch.fill_(float(it))
    torch.cuda.synchronize()
    assert qla.device_status() == 0
    check_all(results, sets, direction, f"{engine} {layout} {direction} thrash={thrash} {release}")


@pytest.mark.parametrize("thrash", [False, True])
@pytest.mark.parametrize("layout,direction", CASES)
@pytest.mark.parametrize("engine", engines_under_test())
def test_in_place_replay(engine, layout, direction, thrash):
    import torch
    if not engine_supports(engine, 128, 128):
        pytest.skip("shape")
    sets = prepare(layout, direction)
    work = [torch.empty_like(s["Hd"]) for s in sets]
    scratch = torch.empty(64 << 20, dtype=torch.float32, device="cuda:0") if thrash else None
    results = []
    for it in range(REPS):
        k = it % 2
        work[k].copy_(sets[k]["Hd"])  # restore H: the previous in-place call overwrote it
        qla.cp_correct(work[k], sets[k]["Md"], sets[k]["h0d"], work[k], layout=layout, direction=direction,
                       engine=engine)
        results.append(work[k].clone())
        if thrash:
            scratch.fill_(float(it))
    torch.cuda.synchronize()
    check_all(results, sets, direction, f"in place {engine} {layout} {direction} thrash={thrash}")


@pytest.mark.parametrize("engine", engines_under_test())
def test_repeated_calls_are_bitwise_identical(engine):
    """Gaussian inputs: the kernels fix their summation order, so repeated
    calls (same arguments, no synchronisation between them) must agree
    bitwise; a race would show as call-to-call differences."""
    import torch
    c = qi.WORKLOADS["c1"]
    H, M, h0 = qi.make_inputs(c, "kv")
    dev = torch.device("cuda:0")
    Hd, Md, h0d = (torch.from_numpy(a).to(dev) for a in (H, M, h0))
    outs = [qla.cp_correct(Hd, Md, h0d, layout="kv", direction="fwd", engine=engine) for _ in range(20)]
    torch.cuda.synchronize()
    first = outs[0].cpu()
    for o in outs[1:]:
        assert torch.equal(o.cpu(), first)
