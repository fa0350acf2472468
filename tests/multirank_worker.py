"""One rank of the CPU (gloo) check of bench.py's multi-rank path, launched
the way torchrun launches bench.py: RANK, WORLD_SIZE, MASTER_ADDR and
MASTER_PORT come from the environment.  Each rank reports made-up step
timings; the rank prints what bench.py would take as the job's timing and
throughput, and what its reference arm does on that rank."""
import contextlib
import io
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    dist.init_process_group("gloo")
    # rank r's timed region took 100 + 7r ms, its end-to-end run 300 - 5r ms
    t_ms, e2e_ms = bench.max_over_ranks(dist, [100.0 + 7 * rank, 300.0 - 5 * rank], "cpu")
    dist.barrier()

    class A:
        steps, warmup, gpus = 2, 3, world

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        ref = bench.run_reference(A, rank, world) if rank != 0 else None
    dist.barrier()
    dist.destroy_process_group()
    print(json.dumps({"rank": rank, "t_ms": t_ms, "e2e_ms": e2e_ms,
                      "value": bench.job_throughput(world, 1e12, 10, t_ms),
                      "reference_stdout": buf.getvalue(), "reference_ret": ref}))


if __name__ == "__main__":
    main()
