"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

Each rank runs its own replica of the workload (weak scaling, no collective
on the data path); the only cross-rank steps are the barrier around the timed
region and the reduction of the step time (max over ranks) and of the bytes
moved (sum over ranks)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r measured 1 + r ms per step and moved (r + 1) GB per step
        ms, rate = bench.job_rate(1.0 + rank, (rank + 1) * 1e9, world, torch.device("cpu"))
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "rate": rate}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_rate_takes_slowest_rank_and_all_bytes(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms"] == pytest.approx(2.0)  # the slowest rank
        assert g["rate"] == pytest.approx(3e9 / 2e-3 / 1e9)  # 3 GB over 2 ms


def test_single_rank_rate_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, rate = bench.job_rate(2.0, 4e9, 1, None)
    assert ms == 2.0 and rate == pytest.approx(2000.0)


def test_replicas_get_their_own_seeds():
    sys.path.insert(0, ROOT)
    import bench
    a, b = bench.make_workload("layout-bs16-scattered", 0), bench.make_workload("layout-bs16-scattered", 1)
    assert a.seq_lens.tolist() == b.seq_lens.tolist()  # same shape of work per rank
    assert not np.array_equal(a.q, b.q)                 # different data
    assert not np.array_equal(a.block_tables, b.block_tables)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
