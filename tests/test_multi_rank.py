"""Multi-rank host logic of the benchmark: world size 2 over gloo, on the CPU.

bench.py runs one process per GPU.  Each rank processes its own shard of the
job (batch element r of a job with B = world; there is no data-path
collective), and rank 0 reports the whole job's figure from the slowest
rank's time.  These tests run those helpers with two gloo ranks on 127.0.0.1:

- the maximum over ranks reaches every rank;
- the shards partition the global job: the oracle's outputs on the two
  shards equal, bitwise, the oracle on the whole B = 2 job;
- the job figure is the slowest rank's time over all ranks' calls;
- the reference arm's non-zero ranks exit at once, without output.
"""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CALLS = 2  # forward kv and forward vk of the bench's step


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory):
    pytest.importorskip("torch.distributed")
    outdir = str(tmp_path_factory.mktemp("ranks"))
    os.environ["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests"),
                                                os.environ.get("PYTHONPATH", "")])
    sys.path[:0] = [p for p in (ROOT, os.path.join(ROOT, "tests")) if p not in sys.path]
    import mr_worker
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=mr_worker.run, args=(r, 2, port, outdir, CALLS)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return outdir


def test_max_over_ranks_reaches_every_rank(two_ranks):
    for r in range(2):
        with open(os.path.join(two_ranks, f"rank{r}.json")) as f:
            d = json.load(f)
        assert d["world"] == 2 and d["max"] == 13.0 and d["ms_slowest"] == 6.0


def test_job_figure_is_slowest_rank_over_all_calls(two_ranks):
    import bench
    with open(os.path.join(two_ranks, "rank0.json")) as f:
        d = json.load(f)
    assert d["job_us"] == pytest.approx(6.0 * 1e3 / (100 * 2))
    assert bench.job_us_per_call(6.0, 100, 1) == pytest.approx(60.0)


def test_shards_partition_the_global_job(two_ranks):
    import bench
    import oracle
    import qla_inputs as qi
    for i, (name, layout, direction) in enumerate(bench.CALLS[:CALLS]):
        whole = qi.WORKLOADS[name].with_(B=2)
        H, M, h0 = qi.make_inputs(whole, layout)
        ref, _ = oracle.cp_correct(H, M, h0, layout, direction)
        for r in range(2):
            got = np.load(os.path.join(two_ranks, f"out_r{r}_c{i}.npy"))
            assert got.shape == ref[r:r + 1].shape
            assert np.array_equal(got, ref[r:r + 1]), f"rank {r} call {name} {layout} {direction}"
    # and the shards differ: rank 1 is not a copy of rank 0
    assert not np.array_equal(np.load(os.path.join(two_ranks, "out_r0_c0.npy")),
                              np.load(os.path.join(two_ranks, "out_r1_c0.npy")))


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
