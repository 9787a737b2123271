"""One rank of the benchmark's multi-rank timing path, for the launcher test.

Started once per rank by bench.launch_ranks (torch.distributed.run) with gloo
instead of NCCL and a fixed per-rank step time in place of the GPU step; rank
0 prints the JSON fields the benchmark derives from the ranks' times: the
world size as n_gpus, the slowest rank's time and the whole-job throughput.
"""
import json
import os
import sys

import torch
import torch.distributed as dist

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

N_PARAMS = 1_000_000


def main():
    world, rank, _ = bench.dist_env()
    dist.init_process_group("gloo")
    try:
        ms = 10.0 + rank  # the last rank is the slowest
        ms = bench.max_over_ranks(ms, world, torch.device("cpu"))
        if rank == 0:
            print(json.dumps({"n_gpus": world, "ms_per_step": ms,
                              "value": bench.replica_throughput(N_PARAMS, world, ms)}), flush=True)
        dist.barrier()
    finally:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
