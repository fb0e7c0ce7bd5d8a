"""bench.py with its measured step replaced by a CPU stand-in.

Used by tests/test_bench_dist.py to run ``--gpus N`` end to end on a machine
without GPUs: the stand-in exercises only the launcher, the gloo process
group and the max-over-ranks reduction; it prints a JSON line of the same
shape whose numbers are the ranks' fake step times, never a measurement.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def stand_in(args, world, rank, local):
    ms = bench.max_over_ranks(1.0 + rank, world)  # rank r "takes" 1 + r ms
    if rank == 0:
        print(json.dumps({"metric": bench.METRIC, "n_gpus": world, "ms_per_step": ms, "stand_in": True}), flush=True)
    return 0


bench.run_ours = stand_in

if __name__ == "__main__":
    sys.exit(bench.main())
