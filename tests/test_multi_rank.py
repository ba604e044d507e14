"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2).

The path shards as independent replicas (no data-path collective): each rank
times its own copy of the workload, the job's time is the slowest rank's
(max over ranks) and the value is the units of all ranks over that time.
The reference arm runs on rank 0 only; the other ranks exit 0 without work.
"""
import json
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
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # each rank reports a different time; every rank must see the largest
        t = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        rate = bench.whole_job_rate(1000.0, world, 4, t)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"t": t, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for g in got:
        assert g["t"] == 15.0
        # 1000 units per rank per step, 2 ranks, 4 steps, over 15 ms
        assert abs(g["rate"] - 1000.0 * 2 * 4 / 15e-3) < 1e-6


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
