"""The N > 1 bench path on the CPU: ranks are independent replicas, the job
time is the slowest rank's time (max over ranks, here over gloo), and the
whole-job throughput counts every rank's tokens."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.reduce_max(1.0 + rank, world)
    q.put((rank, t, bench.aggregate_throughput(world, 120000, 5, t)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_slowest_time_and_sum_tokens():
    world, port = 2, 29617
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]                 # max over ranks
    assert res[0][2] == pytest.approx(2 * 120000 * 5 / 2.0)   # all ranks' tokens


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
