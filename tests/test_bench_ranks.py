"""The replica path of bench.py on the CPU (gloo, world size 2): the timing is
the maximum over ranks and every rank agrees on it; the whole-job value sums the
replicas' work over the slowest replica's time; the oracle arm runs on rank 0
only."""
import json
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
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took 1 + r seconds: every rank must see the slowest, world seconds
    got = bench.max_over_ranks(1.0 + rank, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(got, f)


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        assert json.loads((tmp_path / f"rank{r}.json").read_text()) == float(world)


def test_max_over_ranks_without_group():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


@pytest.mark.parametrize("world", [1, 2, 8])
def test_replica_throughput_is_weak_scaling(world):
    # each replica does the same speed-of-light work per step: the job value
    # grows with the replicas at a fixed slowest-replica time
    one = bench.replica_throughput(1e-3, 10, 1, 0.05)
    assert bench.replica_throughput(1e-3, 10, world, 0.05) == pytest.approx(world * one)
    assert one == pytest.approx(100.0 * 1e-3 * 10 / 0.05)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--gpus", "2"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
