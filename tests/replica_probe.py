"""A rank of the bench's replica launch, run on the CPU: each rank joins a gloo process
group from the torch.distributed.run environment, reports a per-rank step time, and
rank 0 prints the bench's aggregation (max over ranks, whole-job GB/s) as one JSON line.
Used by tests/test_multirank_cpu.py through bench.replica_command."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    try:
        # rank r takes (r + 1) ms per step; the job is as slow as its slowest rank
        ms = bench.max_over_ranks([float(rank + 1)])[0]
        gbs = bench.whole_job_gbs(world, 1_000_000, ms)
        if rank == 0:
            print(json.dumps({"n_gpus": world, "ms_per_step": ms, "value": gbs,
                              "argv": sys.argv[1:]}), flush=True)
        dist.barrier()
    finally:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
