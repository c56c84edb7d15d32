"""The multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1) take the slowest
rank's time, meet at the barrier, and report the whole job's throughput; under a two-rank
launch the reference arm prints one line on rank 0 and nothing on rank 1."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier(world)
        ms = bench.max_over_ranks(1.0 + rank, world)  # rank r took 1 + r ms
        q.put((rank, ms, bench.whole_job_tflops(2e9, world, ms)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, 29517
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, tf in got:
        assert ms == 2.0                      # the slower rank's time on every rank
        assert tf == pytest.approx(2.0)       # 2 ranks x 2 GFLOP in 2 ms = 2 TFLOP/s


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "1", "--oracle-rows", "64"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if rank == 0:
        assert len(lines) == 1 and json.loads(lines[0])["impl"] == "reference"
    else:
        assert lines == []
