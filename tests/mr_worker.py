"""One gloo rank of the multi-rank host tests (started with the spawn method)."""
import json
import os


def run(rank, world, port, outdir, calls):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import numpy as np
    import torch.distributed as dist

    import bench
    import oracle

    r, w, _ = bench.dist_setup(world, backend="gloo")
    got_max = bench.max_over_ranks(10.0 + 3.0 * r, w, device="cpu")
    bench.barrier(w)
    probs = bench.make_problem_set(r)[:calls]
    for i, p in enumerate(probs):
        out, _ = oracle.cp_correct(p["H"], p["M"], p["h0"], p["layout"], p["direction"])
        np.save(os.path.join(outdir, f"out_r{r}_c{i}.npy"), out)
    ms = bench.max_over_ranks(5.0 + r, w, device="cpu")
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "max": got_max, "ms_slowest": ms,
                   "job_us": bench.job_us_per_call(ms, 100, w)}, f)
    dist.destroy_process_group()
