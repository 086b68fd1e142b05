"""Benchmark of the CP state-correction pass on GB300.

Workload: 32 heads, K = V = 128, S = 8 segments (32K tokens at 4K per segment),
fp32 states.  One step is the whole hot path over one batch: four calls of the
C ABI -- forward kv and forward vk on Householder-type M (g (I - beta u u^T)),
reverse kv and reverse vk on M = 0.99 Q (Q Haar-orthogonal) -- each on its own
input set.  The metric is microseconds per call (lower is better), with the
achieved HBM bandwidth of the kernel against the measured copy bandwidth.

Timing: inputs resident in HBM; each step replays a CUDA graph of its four
calls; steps rotate through enough input/output replicas that every call's
buffers were last touched far more than an L2's worth of traffic earlier (the
rotation spans at least 3x the L2 size), so every call reads from DRAM.  Time
is taken with CUDA events on the launching stream, warm-up excluded.

``--impl reference`` times the fp64 CPU oracle instead (the only reference
this computation has), on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADS, K, V, S = 32, 128, 128, 8
CALLS = (("c1", "kv", "fwd"), ("c1", "vk", "fwd"), ("c2", "kv", "rev"), ("c2", "vk", "rev"))
METRIC = "µs per call and achieved HBM GB/s (fraction of roofline) at 32 heads, K=V=128"
WORKLOAD = ("CP state correction, B=1, 32 heads, K=V=128, S=8 (32K tokens / 4K per segment), fp32; "
            "step = fwd kv + fwd vk (Householder M) + rev kv + rev vk (0.99*orthogonal M)")


# GB300's nominal HBM3e bandwidth, for the fraction against the datasheet figure
# beside the one against the measured copy bandwidth.
NOMINAL_HBM_GBS = 8000.0


def algorithmic_bytes(chains, S_, K_, V_, with_init=True):
    """Bytes one call must move: H and M of the S-1 segments it visits, every
    output state, and h_init."""
    return 4 * chains * ((S_ - 1) * K_ * V_ + (S_ - 1) * K_ * K_ + S_ * K_ * V_ + (K_ * V_ if with_init else 0))


def scan_groups(heads, S_, K_, V_):
    """The scan's automatic group count on the current device, read back from
    the library's scratch size (chains x groups x (K^2 + 2 K V) floats)."""
    import linear_attention_context_gb300 as qla
    per_group = heads * (K_ * K_ + 2 * K_ * V_) * 4
    return qla.scan_workspace_bytes(1, heads, S_, K_, V_) // per_group


def algorithmic_flops(chains, S_, K_, V_):
    return 2 * chains * (S_ - 1) * K_ * K_ * V_


def kernel_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    capture, or None when the kernel sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    h = hashlib.sha256()
    for s in d.get("sources", []):
        fp = os.path.join(ROOT, s)
        if not os.path.exists(fp):
            return None
        with open(fp, "rb") as f:
            h.update(f.read())
    return d["dram_bytes_per_launch"] if h.hexdigest() == d.get("sources_sha256") else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def compute_peaks(dev):
    """The two compute ceilings the path could be bound by, on this device:
    dense TF32 tensor throughput, measured (cuBLAS fp32 matmul with TF32
    allowed, 8192^3, best of 5, CUDA events), and the FFMA ceiling computed
    from the SM count (128 fp32 FMA lanes per SM per clock) at the maximum SM
    clock.  Reported beside the HBM roofline."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    n = 8192
    a = torch.randn(n, n, device=dev)
    b = torch.randn(n, n, device=dev)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        for _ in range(2):
            torch.matmul(a, b)
        best = float("inf")
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    del a, b
    max_mhz = 2070.0
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            max_mhz = float(json.load(f).get("sm_max_mhz", max_mhz))
    return {"tf32_tflops": round(2 * n ** 3 / (best * 1e-3) / 1e12, 1),
            "tf32_how": "torch.matmul fp32 8192^3, TF32 allowed, best of 5",
            "ffma_tflops": round(sms * 128 * 2 * max_mhz * 1e6 / 1e12, 1),
            "ffma_how": f"{sms} SMs x 128 FMA/clk x 2 flop x {max_mhz:.0f} MHz",
            "sms": sms, "l2_bytes": props.L2_cache_size}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def mark(self, name):
        self.marks.append((name, time.time()))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0 = dict(self.marks).get("start", 0)
        t1 = dict(self.marks).get("end", time.time())
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ts, ln in self.lines:
            if not (t0 <= ts <= t1 + 0.06):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# Steps captured per CUDA graph in the timed region (rounded to a multiple of
# the replica count).
STEPS_PER_GRAPH = 16


def dist_setup(n_gpus, backend="nccl"):
    """Rank, world size and local rank from the launcher's environment; one
    process per GPU over NCCL (gloo, on the host, for the multi-rank tests)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(ms_slowest, calls_per_rank, world):
    """Whole-job figure: every rank's calls over the slowest rank's time (each
    rank processes its own shard, so the job's calls are world x calls_per_rank)."""
    return ms_slowest * 1e3 / (calls_per_rank * world)


def shard_unit0(rank):
    """First chain of this rank's shard: rank r processes batch element r of a
    job with B = world (the same shapes on every rank, disjoint inputs)."""
    return rank * HEADS


def make_problem_set(rank=0):
    """The four calls' seeded inputs (numpy, host), this rank's shard."""
    import qla_inputs as qi
    probs = []
    for name, layout, direction in CALLS:
        H, M, h0 = qi.make_inputs(qi.WORKLOADS[name], layout, unit0=shard_unit0(rank))
        probs.append(dict(name=name, layout=layout, direction=direction, H=H, M=M, h0=h0))
    return probs


def run_ours(args):
    import numpy as np
    import torch

    import linear_attention_context_gb300 as qla

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    probs = make_problem_set(rank)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_call = sum(p["H"].nbytes * 2 + p["M"].nbytes + p["h0"].nbytes for p in probs) / len(probs)
    reps = max(2, math.ceil(3 * l2 / (per_call * len(probs))))
    bufs = []
    for r in range(reps):
        row = []
        for p in probs:
            row.append(dict(H=torch.from_numpy(p["H"]).to(dev), M=torch.from_numpy(p["M"]).to(dev),
                            h0=torch.from_numpy(p["h0"]).to(dev), out=torch.empty(p["H"].shape, device=dev),
                            layout=p["layout"], direction=p["direction"]))
        bufs.append(row)
    stream = torch.cuda.Stream(dev)
    kw = dict(engine=args.engine, variant=args.variant, release=args.release)
    if args.dependent_launch:
        qla.set_dependent_launch(True)

    def call(b, s=None):
        qla.cp_correct(b["H"], b["M"], b["h0"], b["out"], layout=b["layout"], direction=b["direction"],
                       stream=s, **kw)

    # correctness first (untimed): every replica's outputs against the oracle
    # on the first head (full check happens in the tests)
    with torch.cuda.stream(stream):
        for row in bufs:
            for b in row:
                call(b, stream)
    stream.synchronize()
    if rank == 0 and not args.skip_check:
        import oracle
        from_qla = bufs[0]
        for p, b in zip(probs, from_qla):
            sl = (slice(0, 1), slice(0, 2))
            ref, _ = oracle.cp_correct(p["H"][sl], p["M"][sl], p["h0"][sl], p["layout"], p["direction"])
            got = b["out"][sl].cpu().numpy().astype(np.float64)
            err = np.sqrt(((got - ref) ** 2).sum()) / np.sqrt((ref ** 2).sum())
            if not err <= 1e-5:
                raise SystemExit(f"bench pre-check failed for {p['name']} {p['layout']} {p['direction']}: {err}")

    # CUDA graphs of G consecutive steps (G a multiple of the replica count,
    # so every graph runs the replicas in the same rotation): a graph
    # boundary costs a few microseconds that a long captured sequence does
    # not.  The timed region runs exactly K steps: K // G replays of the
    # G-step graph, then a graph of the K % G remaining steps.
    G = reps * max(1, STEPS_PER_GRAPH // reps)

    def capture(nsteps):
        if nsteps == 0:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in range(nsteps):
                for b in bufs[s % reps]:
                    call(b, stream)
        return g

    with torch.cuda.stream(stream):
        g_full = capture(G)
        g_rest = capture(args.steps % G)
    stream.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        for w in range((args.warmup + G - 1) // G):  # at least W warm-up steps
            g_full.replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark("start")
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps // G):
            g_full.replay()
        if g_rest is not None:
            g_rest.replay()
        e1.record(stream)
    stream.synchronize()
    if sampler:
        sampler.mark("end")
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    clocks = sampler.stop() if sampler else None

    n_calls = args.steps * len(CALLS)
    us_per_call_rank = ms * 1e3 / n_calls
    value = job_us_per_call(ms, n_calls, world)
    var, eng = qla.resolve(1, HEADS, S, K, V, "kv")
    if args.engine != "auto":
        eng = args.engine
    if args.variant != "auto":
        var = args.variant
    launches_per_call = 1 if var == "seq" else 4
    bytes_call = algorithmic_bytes(HEADS, S, K, V)
    achieved = bytes_call / (us_per_call_rank * 1e-6) / 1e9
    peak, peak_kind = load_peaks()

    # end-to-end through the public API with host buffers: pinned host inputs
    # copied in and outputs copied out inside the timed region
    e2e = None
    if not args.skip_e2e:
        hin = [dict(H=torch.from_numpy(p["H"]).pin_memory(), M=torch.from_numpy(p["M"]).pin_memory(),
                    h0=torch.from_numpy(p["h0"]).pin_memory(), out=torch.empty(p["H"].shape).pin_memory())
               for p in probs]
        e2e_steps = max(3, min(args.steps, 50))
        # Copies overlap compute as a user would pipeline them: inputs of a
        # call go up on one stream, calls run on another, results come down on
        # a third; each call's device buffers are reused two steps later (the
        # replicas), once that earlier call's kernel and result copy are done.
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        nb = 2

        def e2e_run(nsteps):
            ev = lambda: torch.cuda.Event()  # noqa: E731
            comp_done, out_done = {}, {}
            for n in range(nsteps * len(CALLS)):
                st, kind = divmod(n, len(CALLS))
                b, h = bufs[st % nb][kind], hin[kind]
                with torch.cuda.stream(s_in):
                    if n - nb * len(CALLS) in comp_done:
                        s_in.wait_event(comp_done[n - nb * len(CALLS)])
                    b["H"].copy_(h["H"], non_blocking=True)
                    b["M"].copy_(h["M"], non_blocking=True)
                    b["h0"].copy_(h["h0"], non_blocking=True)
                    e_in = ev()
                    e_in.record(s_in)
                with torch.cuda.stream(stream):
                    stream.wait_event(e_in)
                    if n - nb * len(CALLS) in out_done:
                        stream.wait_event(out_done[n - nb * len(CALLS)])
                    call(b, stream)
                    comp_done[n] = ev()
                    comp_done[n].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[n])
                    h["out"].copy_(b["out"], non_blocking=True)
                    out_done[n] = ev()
                    out_done[n].record(s_out)
            return out_done[nsteps * len(CALLS) - 1]

        last = e2e_run(3)
        torch.cuda.synchronize()
        barrier(world)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for si in (s_in, s_out):
            si.wait_event(a0)
        last = e2e_run(e2e_steps)
        stream.wait_event(last)
        a1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(a0.elapsed_time(a1), world)
        h2d = sum(h["H"].nbytes + h["M"].nbytes + h["h0"].nbytes for h in hin)
        d2h = sum(h["out"].nbytes for h in hin)
        e2e = {"value": round(job_us_per_call(ems, e2e_steps * len(CALLS), world), 3), "unit": "us",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peaks = compute_peaks(dev) if rank == 0 and not args.skip_peaks else None
    cpu = None
    if rank == 0 and not args.skip_cpu:
        cpu = cpu_baseline(probs, budget_s=args.cpu_budget)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "us", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; Householder and 0.99*orthogonal M, N(0,1)*0.1 states)",
            "config": {"workload": WORKLOAD, "B": 1, "heads": HEADS, "K": K, "V": V, "S": S,
                       "calls_per_step": len(CALLS), "variant": var, "engine": eng, "release": args.release,
                       "l2_defeat": f"inputs larger than L2: {reps} rotating replicas x {len(CALLS)} calls "
                                    f"({reps * len(CALLS) * per_call / 1e6:.0f} MB) vs L2 {l2 / 1e6:.0f} MB",
                       "graph": f"CUDA graphs of {G} steps ({G * len(CALLS)} calls) replayed back to back",
                       "dependent_launch": bool(args.dependent_launch),
                       "parallelism": f"replicas x{world} (no collective)"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS,
                         "traffic": args.traffic if args.traffic is not None else (kernel_traffic() if eng == "tc" else None),
                         "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                                        if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "algorithmic_bytes_per_launch": bytes_call, "launches_per_call": launches_per_call,
                         "avg_launch_us": round(us_per_call_rank / launches_per_call, 3),
                         "flops_per_call": algorithmic_flops(HEADS, S, K, V)},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": n_calls * launches_per_call, "clocks": clocks,
        }
        if peaks:
            # the tensor-pipe view of the same calls: 3xTF32 executes 3x the algorithmic flops
            executed = 3 * algorithmic_flops(HEADS, S, K, V) if eng == "tc" else algorithmic_flops(HEADS, S, K, V)
            rate = executed / (us_per_call_rank * 1e-6) / 1e12
            ceiling = peaks["tf32_tflops"] if eng == "tc" else peaks["ffma_tflops"]
            line["compute"] = {"executed_tflops": round(rate, 1),
                               "ceiling_tflops": ceiling,
                               "ceiling": "tf32 tensor (measured)" if eng == "tc" else "ffma (computed)",
                               "frac": round(rate / ceiling, 4), "peaks": peaks}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cpu_baseline(probs, budget_s=20.0):
    """The oracle as it stands, on this host's cores, on the same four calls.
    Runs whole calls (all 32 heads) when they fit the budget, else a head
    sample; returns microseconds per full call."""
    import oracle
    t0 = time.perf_counter()
    p = probs[0]
    _, _, threads = oracle.cp_correct(p["H"][:, :1], p["M"][:, :1], p["h0"][:, :1], p["layout"], p["direction"],
                                      return_threads=True)
    per_head = time.perf_counter() - t0  # single head, one thread busy
    heads = HEADS
    est = per_head * HEADS * len(probs) / max(1, min(threads, HEADS))
    if est > budget_s:
        heads = max(threads, int(HEADS * budget_s / est))
        heads = min(HEADS, heads)
    t = time.perf_counter()
    for q in probs:
        oracle.cp_correct(q["H"][:, :heads], q["M"][:, :heads], q["h0"][:, :heads], q["layout"], q["direction"])
    el = time.perf_counter() - t
    us_per_call = el / len(probs) * (HEADS / heads) * 1e6
    # the same oracle on one thread: two heads of each call, scaled to a full call
    t = time.perf_counter()
    for q in probs:
        oracle.cp_correct(q["H"][:, :2], q["M"][:, :2], q["h0"][:, :2], q["layout"], q["direction"], nthreads=1)
    one = (time.perf_counter() - t) / len(probs) * (HEADS / 2) * 1e6
    return {"value": round(us_per_call, 1), "unit": "us", "cores": threads, "kind": "oracle",
            "sample": f"{len(probs)} calls x {heads} of {HEADS} heads (fp64 oracle, {threads} threads), "
                      f"scaled to a full call",
            "single_thread": {"value": round(one, 1), "unit": "us",
                              "sample": f"{len(probs)} calls x 2 of {HEADS} heads on one thread, scaled"}}


def run_reference(args):
    """The oracle timed as the reference arm: K steps after W warm-up steps,
    each step one bounded sample (a block of heads of one of the four calls,
    rotating), reported per full call."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    probs = make_problem_set()
    # calibrate: one head of one call
    p = probs[0]
    t0 = time.perf_counter()
    _, _, threads = oracle.cp_correct(p["H"][:, :1], p["M"][:, :1], p["h0"][:, :1], p["layout"], p["direction"],
                                      return_threads=True)
    one = time.perf_counter() - t0  # one head on one thread
    # Each step runs a multiple of the thread count in heads (the oracle's
    # threads take one head each), as many rounds as the per-step budget allows.
    budget = 150.0 / max(1, args.steps + args.warmup)
    rounds = max(1, int(budget / max(one, 1e-9)))
    heads = max(1, min(HEADS, threads * rounds))
    cores = min(threads, heads)
    times = []
    for s in range(args.warmup + args.steps):
        q = probs[s % len(probs)]
        t = time.perf_counter()
        oracle.cp_correct(q["H"][:, :heads], q["M"][:, :heads], q["h0"][:, :heads], q["layout"], q["direction"])
        if s >= args.warmup:
            times.append(time.perf_counter() - t)
    total = sum(times)
    us_per_call = total / len(times) * (HEADS / heads) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": round(us_per_call, 1), "unit": "us", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; same inputs as the GPU arm)",
            "config": {"workload": WORKLOAD, "B": 1, "heads": HEADS, "K": K, "V": V, "S": S,
                       "calls_per_step": 1, "parallelism": "host threads"},
            "cpu_baseline": {"value": round(us_per_call, 1), "unit": "us", "cores": cores, "kind": "oracle",
                             "sample": f"each step: {heads} of {HEADS} heads of one call (rotating over the "
                                       f"4 calls), scaled to a full call"},
            "e2e": {"value": round(us_per_call, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """Low batch*heads sweep (B=1, K=V=128, 0.99*orthogonal M): the sequential
    kernel against the group scan, per (heads, S), forward kv and reverse vk.
    One JSON line per point; not the headline metric."""
    import torch

    import linear_attention_context_gb300 as qla
    import qla_inputs as qi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream(dev)
    lines = []
    points = [(h, s_) for h in qi.SWEEP_HEADS for s_ in qi.SWEEP_S]
    if args.sweep_point:
        h, s_ = (int(x) for x in args.sweep_point.split(","))
        points = [(h, s_)]
    for heads, S_ in points:
        c = qi.sweep_case(heads, S_)
        for layout, direction in (("kv", "fwd"), ("vk", "rev")):
            H, M, h0 = qi.make_inputs(c, layout)
            Hd, Md, h0d = (torch.from_numpy(a).to(dev) for a in (H, M, h0))
            out = torch.empty_like(Hd)
            times = {}
            for variant in ("seq", "scan"):
                def call():
                    qla.cp_correct(Hd, Md, h0d, out, layout=layout, direction=direction, variant=variant,
                                   stream=stream)
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        call()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for _ in range(10):
                            call()
                stream.synchronize()
                with torch.cuda.stream(stream):  # warm-up replays on the timed stream
                    for _ in range(3):
                        g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    for _ in range(args.sweep_reps):
                        g.replay()
                    e1.record(stream)
                stream.synchronize()
                times[variant] = e0.elapsed_time(e1) * 1e3 / (10 * args.sweep_reps)
            auto = qla.resolve(1, heads, S_, 128, 128, layout)[0]
            # the scan's executed tensor work (3xTF32: 3x) per chain: group
            # products of M, S steps of K^3; group recurrences (S steps),
            # carries (G) and re-runs (S - G), K^2 V each
            Kk = Vv = 128
            G = scan_groups(heads, S_, Kk, Vv)
            flops = 3 * 2 * heads * (S_ * Kk ** 3 + 2 * S_ * Kk * Kk * Vv)
            rate = flops / (times["scan"] * 1e-6) / 1e12
            lines.append({"sweep": {"heads": heads, "S": S_, "layout": layout, "direction": direction},
                          "us_per_call": {k: round(v, 2) for k, v in times.items()},
                          "auto": auto, "bytes_per_call": algorithmic_bytes(heads, S_, 128, 128),
                          "scan_tensor": {"groups": G, "executed_tflops": round(rate, 1)}})
    # the matmul peak last: its power draw would lower the clocks of the timings
    peaks = compute_peaks(dev)
    print(json.dumps({"compute_peaks": peaks}), flush=True)
    for ln in lines:
        ln["scan_tensor"]["frac_of_tf32"] = round(ln["scan_tensor"]["executed_tflops"] / peaks["tf32_tflops"], 4)
        print(json.dumps(ln), flush=True)


def run_varlen(args):
    """Variable-length calls (K=V=128, Householder M): sequences of different
    segment counts packed along the segment axis, the sequential variant
    against the group scan.  One JSON line per case; not the headline metric."""
    import numpy as np
    import torch

    import linear_attention_context_gb300 as qla
    import qla_inputs as qi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream(dev)
    cases = [  # (lengths, heads)
        ([128, 37, 0, 90], 1),
        ([64, 64], 2),
        ([200, 3, 17, 41, 9, 0, 120, 8], 1),
        ([8] * 32, 32),
    ]
    for lengths, heads in cases:
        H, M, h0, cu = qi.make_varlen_inputs(lengths, heads, 128, 128, seed=51, m_kind="householder",
                                             h_scale=0.1, init_scale=0.1)
        Hd, Md, h0d = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (H, M, h0))
        cud = torch.from_numpy(cu.astype(np.int32)).to(dev)
        out = torch.empty_like(Hd)
        bound = max(lengths)
        times = {}
        for variant in ("seq", "scan"):
            def call():
                qla.cp_correct_varlen(Hd, Md, cud, h0d, out, variant=variant, max_segments=bound, stream=stream)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    call()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(10):
                        call()
            stream.synchronize()
            with torch.cuda.stream(stream):  # warm-up replays on the timed stream
                for _ in range(3):
                    g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(args.sweep_reps):
                    g.replay()
                e1.record(stream)
            stream.synchronize()
            times[variant] = e0.elapsed_time(e1) * 1e3 / (10 * args.sweep_reps)
        print(json.dumps({"varlen": {"lengths": lengths, "heads": heads, "K": 128, "V": 128},
                          "us_per_call": {k: round(v, 2) for k, v in times.items()}}), flush=True)
    if qla.device_status() != 0:
        raise SystemExit("device status word set during the varlen timings")


def run_configs(args):
    """Configs 0-2 one at a time (config 3: --large, config 4: --sweep): µs per
    call of each (layout, direction) of the config, graph-replayed, L2 flushed
    by rotating input copies where the inputs are smaller than L2.  One JSON
    line per config; not the headline metric."""
    import numpy as np
    import torch

    import linear_attention_context_gb300 as qla
    import qla_inputs as qi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream(dev)
    peak, peak_source = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    plan = {"c0": [("kv", "fwd")], "c1": [("kv", "fwd"), ("vk", "fwd")], "c2": [("kv", "rev"), ("vk", "rev")]}
    for name, combos in plan.items():
        c = qi.WORKLOADS[name]
        times = {}
        for layout, direction in combos:
            H, M, h0 = qi.make_inputs(c, layout)
            per_set = H.nbytes + M.nbytes + (h0.nbytes if h0 is not None else 0) + H.nbytes
            nsets = max(1, min(16, int(np.ceil(2 * l2 / per_set))))
            sets = []
            for _ in range(nsets):
                sets.append((torch.from_numpy(H).to(dev), torch.from_numpy(M).to(dev),
                             None if h0 is None else torch.from_numpy(h0).to(dev), torch.empty(H.shape, dtype=torch.float32, device=dev)))
            calls = 16 * nsets

            def body():
                for _ in range(16):
                    for Hd, Md, h0d, out in sets:
                        qla.cp_correct(Hd, Md, h0d, out, layout=layout, direction=direction, stream=stream,
                                       engine=args.engine)
            with torch.cuda.stream(stream):
                body()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    body()
            stream.synchronize()
            with torch.cuda.stream(stream):  # warm-up replays on the timed stream
                for _ in range(3):
                    g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(args.sweep_reps):
                    g.replay()
                e1.record(stream)
            stream.synchronize()
            times[f"{layout} {direction}"] = e0.elapsed_time(e1) * 1e3 / (calls * args.sweep_reps)
        us = float(np.mean(list(times.values())))
        b = algorithmic_bytes(c.B * c.heads, c.S, c.K, c.V, with_init=c.init_kind != "none")
        line = {"config": name, "B": c.B, "heads": c.heads, "K": c.K, "V": c.V, "S": c.S,
                "us_per_call": {k: round(v, 3) for k, v in times.items()}, "mean_us": round(us, 3),
                "engine": args.engine if args.engine != "auto" else qla.resolve(c.B, c.heads, c.S, c.K, c.V)[1],
                "algorithmic_bytes": b,
                "hbm_gbs": round(b / (us * 1e-6) / 1e9, 1)}
        line["hbm_frac"] = round(b / (us * 1e-6) / 1e9 / peak, 4)
        line["peak"] = f"{peak} GB/s ({peak_source})"
        rot = per_set * len(sets)
        line["l2"] = (f"{len(sets)} rotating input/output sets, {rot / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB"
                      + ("" if rot >= 2 * l2 else " (the sets fit in L2: inputs partly L2-resident)"))
        print(json.dumps(line), flush=True)


def run_large(args):
    """The 4 x 64-head, K=V=256, S=32 workload (6.4 GB of states), forward
    and reverse kv: one call at a time, CUDA events, after two warm-up calls.
    Not the headline metric."""
    import torch

    import linear_attention_context_gb300 as qla
    import qla_inputs as qi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    c = qi.WORKLOADS["c3"]
    H, M, h0 = qi.make_inputs(c, "kv")
    Hd, Md, h0d = (torch.from_numpy(a).to(dev) for a in (H, M, h0))
    del H, M
    out = torch.empty_like(Hd)
    peak, _ = load_peaks()
    nbytes = algorithmic_bytes(c.chains, c.S, c.K, c.V)
    for direction in ("fwd", "rev"):
        for _ in range(2):
            qla.cp_correct(Hd, Md, h0d, out, layout="kv", direction=direction)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record()
        for _ in range(reps):
            qla.cp_correct(Hd, Md, h0d, out, layout="kv", direction=direction)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        print(json.dumps({"large": {"B": c.B, "heads": c.heads, "K": c.K, "V": c.V, "S": c.S, "layout": "kv",
                                    "direction": direction},
                          "us_per_call": round(us, 1), "gbs": round(nbytes / us / 1e3, 1),
                          "frac_of_measured_hbm": round(nbytes / us / 1e3 / peak, 4),
                          "algorithmic_bytes": nbytes, "variant_engine": qla.resolve(c.B, c.heads, c.S, c.K, c.V)}),
              flush=True)


def local_flops(chains, T, K_, V_):
    """FFMA flops of the local pass: per token and column of [H | M], a dot
    product and an update over the K rows."""
    return 4 * chains * T * K_ * (K_ + V_)


def run_local(args):
    """The per-segment local pass that produces (H_i, M_i) from token-level
    inputs (gated delta rule), on 32 heads x 32K tokens in 8 segments of 4K,
    K = V = 128: its time against the FFMA ceiling, then the local pass and the
    forward correction chained on one stream (the correction launched as a
    programmatic dependent), replayed in a CUDA graph.  The inputs (537 MB of
    bf16 keys and values) exceed L2.  One head of the outputs is checked
    against the fp64 oracle.  One JSON line; not the headline metric."""
    import numpy as np
    import torch

    import linear_attention_context_gb300 as qla
    import oracle
    import qla_inputs as qi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream(dev)
    c = qi.LOCAL_WORKLOADS["l1"]
    k, v, b, g = qi.make_local_inputs(c)
    dk, dv, db, dg = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (k, v, b, g))
    H = torch.empty((c.B, c.heads, c.S, c.K, c.V), device=dev)
    M = torch.empty((c.B, c.heads, c.S, c.K, c.K), device=dev)
    out = torch.empty_like(H)
    h0 = torch.zeros((c.B, c.heads, c.K, c.V), device=dev)
    peaks = compute_peaks(dev) if not args.skip_peaks else None
    ffma = peaks["ffma_tflops"] if peaks else 80.5

    def timed(fn, reps):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                fn()
        stream.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(3):
                gr.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                gr.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    def local():
        qla.local_pass(dk, dv, db, dg, c.S, H, M, stream=stream)

    def chained():
        qla.local_pass(dk, dv, db, dg, c.S, H, M, stream=stream)
        qla.cp_correct(H, M, h0, out, variant="seq", stream=stream)

    us_local = timed(local, args.sweep_reps)
    qla.set_dependent_launch(True)
    try:
        us_pair = timed(chained, args.sweep_reps)
    finally:
        qla.set_dependent_launch(False)
    # check one head of H, M and the corrected states against the oracle
    sl = (slice(0, 1), slice(0, 1))
    Hr, Mr = oracle.local_pass(k[sl], v[sl], b[sl], g[sl], c.S)
    ref, _ = oracle.cp_correct(Hr.astype(np.float32), Mr.astype(np.float32), np.zeros((1, 1, c.K, c.V), np.float32),
                               "kv", "fwd")
    err = {}
    for name, got, r in (("H", H, Hr), ("M", M, Mr), ("out", out, ref)):
        gg = got[0:1, 0:1].cpu().numpy().astype(np.float64)
        d = (gg - r).reshape(c.S, -1)
        err[name] = float(np.max(np.linalg.norm(d, axis=1) / np.maximum(np.linalg.norm(r.reshape(c.S, -1), axis=1),
                                                                           1e-300)))
    if max(err.values()) > 1e-5:
        raise SystemExit(f"local pass outside the parity bar: {err}")
    flops = local_flops(c.chains, c.T, c.K, c.V)
    rate = flops / (us_local * 1e-6) / 1e12
    line = {"local_pass": {"workload": f"B=1, {c.heads} heads, {c.T} tokens in {c.S} segments of {c.L}, "
                                       f"K=V={c.K}, bf16 keys/values, fp32 states", "layout": "kv"},
            "us_per_call": round(us_local, 1),
            "roofline": {"bound": "alu", "achieved": round(rate, 2), "peak": ffma, "unit": "TFLOP/s",
                         "frac": round(rate / ffma, 4), "flops_per_call": flops,
                         "peak_source": "FFMA: SMs x 128 FMA/clk x 2 x max SM clock"},
            "chained_with_correction_us": round(us_pair, 1),
            "correction_share_us": round(us_pair - us_local, 1),
            "max_rel_l2_one_head": {k_: float(f"{v_:.3e}") for k_, v_ in err.items()},
            "input_bytes": int(k.nbytes + v.nbytes + b.nbytes + g.nbytes)}
    print(json.dumps(line), flush=True)
    if qla.device_status() != 0:
        raise SystemExit("device status word set during the local-pass timings")


def run_accuracy(args):
    """Worst per-state error against the fp64 oracle, config by config, with
    the library's automatic choices (configs 0-3 in full; config 4 at its
    sweep points, both layouts and directions).  One JSON line per case."""
    import numpy as np
    import torch

    import linear_attention_context_gb300 as qla
    import oracle
    import qla_inputs as qi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)

    def worst(got, ref):
        g = got.reshape(-1, got.shape[-2] * got.shape[-1]).astype(np.float64)
        r = ref.reshape(g.shape)
        d = g - r
        rel = np.linalg.norm(d, axis=1) / np.maximum(np.linalg.norm(r, axis=1), 1e-300)
        rmax = np.abs(d).max(axis=1) / np.maximum(np.abs(r).max(axis=1), 1e-300)
        return float(rel.max()), float(rmax.max())

    def case(name, c, layout, direction):
        H, M, h0 = qi.make_inputs(c, layout)
        Hd, Md = torch.from_numpy(H).to(dev), torch.from_numpy(M).to(dev)
        h0d = None if h0 is None else torch.from_numpy(h0).to(dev)
        out = qla.cp_correct(Hd, Md, h0d, layout=layout, direction=direction)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        del out, Hd, Md
        rel = rmax = 0.0
        n = c.chains
        flat = lambda a: a.reshape((1, n) + a.shape[2:])  # noqa: E731
        for c0 in range(0, n, 32):  # the oracle in blocks of chains
            sl = (slice(None), slice(c0, min(n, c0 + 32)))
            ref, _ = oracle.cp_correct(flat(H)[sl], flat(M)[sl], None if h0 is None else flat(h0)[sl], layout,
                                       direction)
            a, b = worst(flat(got)[sl], ref)
            rel, rmax = max(rel, a), max(rmax, b)
        v, e = qla.resolve(c.B, c.heads, c.S, c.K, c.V, layout)
        print(json.dumps({"accuracy": name, "B": c.B, "heads": c.heads, "K": c.K, "V": c.V, "S": c.S,
                          "layout": layout, "direction": direction, "variant": v, "engine": e,
                          "worst_rel_l2": float(f"{rel:.3e}"), "worst_rel_max": float(f"{rmax:.3e}")}), flush=True)

    for name, combos in (("c0", [("kv", "fwd")]), ("c1", [("kv", "fwd"), ("vk", "fwd")]),
                         ("c2", [("kv", "rev"), ("vk", "rev")]), ("c3", [("kv", "fwd"), ("kv", "rev")])):
        for layout, direction in combos:
            case(name, qi.WORKLOADS[name], layout, direction)
    for heads in qi.SWEEP_HEADS:
        for S_ in qi.SWEEP_S:
            for layout in ("kv", "vk"):
                for direction in ("fwd", "rev"):
                    case("c4", qi.sweep_case(heads, S_), layout, direction)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--engine", default="auto")
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--release", default="membar")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the current kernel build (read+write)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-check", action="store_true")
    ap.add_argument("--skip-peaks", action="store_true", help="skip the TF32 matmul peak measurement")
    ap.add_argument("--sweep", action="store_true", help="time sequential vs scan over the low batch*heads sweep")
    ap.add_argument("--sweep-reps", type=int, default=20)
    ap.add_argument("--sweep-point", default="", help="heads,S: one point of the sweep only")
    ap.add_argument("--large", action="store_true", help="time the 4 x 64-head K=V=256 S=32 workload")
    ap.add_argument("--varlen", action="store_true", help="time variable-length calls, sequential vs scan")
    ap.add_argument("--configs", action="store_true", help="time configs 0-2 one at a time")
    ap.add_argument("--local", action="store_true", help="time the per-segment local pass and its chain into the correction")
    ap.add_argument("--accuracy", action="store_true", help="worst per-state error against the oracle, per config")
    ap.add_argument("--dependent-launch", action="store_true",
                    help="launch every correction call as a programmatic dependent of the previous one")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.large:
        run_large(args)
    elif args.varlen:
        run_varlen(args)
    elif args.local:
        run_local(args)
    elif args.accuracy:
        run_accuracy(args)
    elif args.configs:
        run_configs(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
