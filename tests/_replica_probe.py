"""One replica of the bench's multi-process launch, on the CPU (gloo): used by
tests/test_bench_dist.py to run the torchrun command line that bench.py
builds for ``--gpus N``."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bench  # noqa: E402


def main():
    torch.distributed.init_process_group("gloo")
    bench._dist = True
    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    bench.barrier()
    worst = bench.dist_max(1.0 + rank)
    if rank == 0:
        print(json.dumps({"world": world, "worst_ms": worst,
                          "value": bench.whole_job_tflops(1e12, world, worst), "argv": sys.argv[1:]}))
    torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
