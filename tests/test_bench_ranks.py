"""The host side of bench.py under torchrun, on CPU: two gloo ranks (one process per GPU in
the real run) each time their own batch; the whole job's time is the slowest rank's and its
throughput counts every rank's units.  No GPU is involved."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        dist.barrier()
        out.put((rank, ms, bench.whole_job_rate(640, world, 10, ms)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_slowest_rank_sets_the_whole_job_rate(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [12.5, 20.0]                        # ms per rank for 10 steps of 640 query-layers
    port = 29500 + os.getpid() % 2000
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in res:
        assert ms == max(times)                 # every rank sees the slowest rank's time
        assert rate == pytest.approx(640 * world * 10 / (max(times) / 1000.0))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_rate(640, 1, 2000, 1000.0) == pytest.approx(640 * 2000)


def test_reference_arm_prints_on_rank_zero_only():
    # under torchrun the reference arm (the CPU oracle) runs on rank 0 alone; other ranks exit 0
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
