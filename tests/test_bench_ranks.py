"""bench.py's multi-rank host logic on CPU: world_size-2 gloo ranks agree on the
slowest rank's time, the whole-job value is weak-scaled from it, and the
reference arm runs on rank 0 alone (the other ranks exit at once)."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as tdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 7.5][rank]                      # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, "cpu")
        gbs = bench.whole_job_gbs(1e9, world, ms)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{ms!r} {gbs!r}")
    finally:
        tdist.destroy_process_group()


def test_ranks_agree_on_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    got = [tuple(map(float, open(tmp_path / f"r{r}.txt").read().split())) for r in range(world)]
    for ms, gbs in got:
        assert ms == 7.5
        assert gbs == pytest.approx(2 * 1e9 / 7.5e-3 / 1e9)


def test_single_process_is_unchanged():
    assert bench.max_over_ranks(4.25) == 4.25
    assert bench.whole_job_gbs(2e9, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
