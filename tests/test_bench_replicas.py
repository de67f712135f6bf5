"""The bench's replica path on CPU: two gloo ranks agree on the slowest rank's
time, the whole-job value counts every replica's work, and under torchrun the
reference arm runs on rank 0 only (the others exit 0 without output)."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank            # this rank's timed milliseconds
        got = bench.max_over_ranks(mine, dist, "cpu")
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr(got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    vals = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(world)]
    assert vals == [15.0, 15.0]


def test_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    f = bench.STEP_FLOPS
    one = bench.job_tflops(1, f, 3, 15.0)
    assert one == pytest.approx(f * 3 / 0.015 / 1e12)
    assert bench.job_tflops(2, f, 3, 15.0) == pytest.approx(2 * one)
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_recorded_counters_follow_code_not_comments():
    """The digest that keeps roofline.traffic tied to the sources it was measured
    on ignores comments and layout but not code."""
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) {\n    return x + 1;   // one more\n}\n"
    b = "/* header */ int f(int x) { return x + 1; }"
    c = "int f(int x) { return x + 2; }"
    assert bench.source_code_only(a) == bench.source_code_only(b)
    assert bench.source_code_only(a) != bench.source_code_only(c)
