"""A stand-in for ``bench.py`` used by tests/test_dist_gloo.py: the bench's
own main() (argument handling, the replica launcher, the process group,
max-over-ranks and the job throughput), with the GPU legs replaced by a
CPU step, so that ``--gpus 2`` can run as two gloo ranks on a machine with no
GPU.  Not a test module (pytest does not collect it)."""
import json
import sys
import time
from pathlib import Path

sys.path.insert(0, str(Path(__file__).resolve().parent.parent))

import bench  # noqa: E402


def cpu_legs(args, rank, world, local):
    bench.barrier(world)
    t0 = time.perf_counter()
    time.sleep(0.05 * (rank + 1))  # rank 1 is the slow one
    seconds = bench.max_over_ranks(time.perf_counter() - t0, world)
    bench.barrier(world)
    if rank == 0:
        print(json.dumps({"metric": bench.METRIC, "n_gpus": world, "steps": args.steps,
                          "value": bench.job_throughput(world, 1000.0 * args.steps, seconds),
                          "seconds": seconds, "local_rank": local}), flush=True)


bench.run_ours = cpu_legs

if __name__ == "__main__":
    bench.main()
