"""Host logic of bench.py's multi-rank (replicas) path, on CPU with gloo.

The GPU arm runs one replica of the workload per rank and reports the units
of all ranks over the slowest rank's time; the reference arm runs on rank 0
only. These tests cover that logic with two gloo ranks; no GPU is used.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank 1 is the slow one on the first value, rank 0 on the second
    ms = [1.0 + rank, 5.0 - rank]
    got = bench.max_over_ranks(ms, world)
    value, unit = bench.value_of("decode", 1e9 * world, got[0])
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got, "value": value, "unit": unit}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max"] == [2.0, 5.0]  # per-value maximum over the ranks
        # whole-job throughput: both ranks' units over the slowest rank's time
        assert r["value"] == pytest.approx(2e9 / 2e-3 / 1e9)
        assert r["unit"] == "GB/s"


def test_max_over_ranks_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3, 4.5], 1) == [3.0, 4.5]


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


@pytest.mark.parametrize("args", [
    ["--workload", "causal_prefill", "--num-splits", "4"],   # a prefill workload
    ["--workload", "paged_decode", "--num-splits", "4"],     # the paged decode: default plan only
    ["--workload", "long_decode", "--num-splits", "-1"],
    ["--warmup", "2"],
])
def test_bench_rejects_bad_options(args):
    """Argument errors end the bench before any GPU work (exit status 2)."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 2, r.stderr
    assert "error:" in r.stderr
