"""The N > 1 host logic of bench.py, on the CPU with two gloo ranks: each rank runs its
own batch (replicas, weak scaling), the job's step time is the slowest rank's, and the
job's throughput counts the units of every rank.  The reference arm runs on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    from structured_mask_linear_gb300.inputs import make_inputs, workload

    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.job_time(1.5 + rank, world, dist, torch.device("cpu"))
    value = bench.job_value(4 * 8192, world, ms)
    w = workload("tiny")
    x = make_inputs(w, "cpu", seed=rank)  # bench.py seeds each replica by its rank
    digest = float(x.q.double().sum())
    got = [None] * world
    dist.all_gather_object(got, digest)
    dist.destroy_process_group()
    with open(os.path.join(out, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value, "digests": got}, f)


def test_two_rank_timing_and_replica_inputs(tmp_path):
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["ms"] == 2.5  # max over ranks, seen by every rank
        assert r["value"] == pytest.approx(2 * 4 * 8192 / 2.5e-3)
    assert res[0]["digests"] == res[1]["digests"]
    assert res[0]["digests"][0] != res[0]["digests"][1]  # replicas draw different inputs


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_time(3.25, 1) == 3.25
    assert bench.job_value(100, 1, 2.0) == pytest.approx(5e4)


def test_reference_arm_other_ranks_exit_without_output():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0
    assert p.stdout.strip() == ""
