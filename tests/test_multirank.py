"""The multi-rank host logic of bench.py on CPU: two gloo ranks (no GPU).

Every rank runs an independent replica of the workload (the path has no
exchange step, so there is no collective on the data path); the step time is
the max over ranks and the value counts the units of all ranks.  The
reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r "measured" 1.5 + r ms per step
    ms = bench.max_over_ranks(1.5 + rank, world, "cpu")
    rate = bench.whole_job_rate(1000.0, ms, world)
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms} {rate} {int(bench.reference_runs_on(rank))}\n")
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_value(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for r, (ms, rate, ref) in enumerate(rows):
        assert float(ms) == pytest.approx(2.5)                 # the slowest rank's time
        assert float(rate) == pytest.approx(2 * 1000.0 / 2.5e-3)   # both ranks' units
        assert int(ref) == (1 if r == 0 else 0)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.whole_job_rate(500.0, 2.0, 1) == pytest.approx(250000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"],
                       env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
