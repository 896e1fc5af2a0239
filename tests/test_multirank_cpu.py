"""The bench's N>1 path (replicas: one pack per GPU, no data-path collective) on CPU:
two gloo ranks check the max-over-ranks timing and the whole-job throughput."""
import os

import pytest
import torch.multiprocessing as mp

import bench


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r+1) ms per step; the job is as slow as its slowest rank
        vals = bench.max_over_ranks([10.0 * (rank + 1), 4.0 + rank, 6.0 * (rank + 1)])
        gbs = bench.whole_job_gbs(world, 1_000_000, vals[0] / 10)
        q.put((rank, vals, gbs))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, vals, gbs in res:
        assert vals == [20.0, 5.0, 12.0]
        # 2 ranks x 1 MB per step over the slowest rank's 2 ms
        assert gbs == pytest.approx(2 * 1_000_000 / 2e-3 / 1e9)


def test_single_rank_is_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.whole_job_gbs(1, 2_000_000, 1.0) == pytest.approx(2.0)


def test_replica_launch_end_to_end():
    """The command bench.py runs for --gpus N without a torchrun environment starts N
    ranks of one node on 127.0.0.1; run here with a CPU probe as the script, the ranks
    rendezvous, aggregate over all of them, and rank 0 alone prints the line."""
    import json
    import subprocess
    probe = os.path.join(os.path.dirname(os.path.abspath(__file__)), "replica_probe.py")
    cmd = bench.replica_command(probe, ["--gpus", "2", "--steps", "3"], 2, bench.free_port())
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=180, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2 and out["ms_per_step"] == 2.0
    assert out["value"] == pytest.approx(2 * 1_000_000 / 2e-3 / 1e9)
    assert out["argv"] == ["--gpus", "2", "--steps", "3"]
