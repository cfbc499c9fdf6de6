"""The N > 1 path of bench.py on the CPU: two gloo ranks, replicas only.

The layer shards by token tiles with no exchange, so bench.py runs one replica
per GPU; the process group only lines the ranks up and takes the slowest rank's
time.  These tests run that logic with world size 2 over gloo (127.0.0.1)."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        rep = bench.Replicas(world, "cpu")
        rep.barrier()
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
        worst = rep.max(local_ms)
        rep.barrier()
        value = bench.job_throughput(8192, 3, world, worst)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"worst": worst, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert res[0] == res[1]
    assert res[0]["worst"] == 15.0
    # whole-job throughput: both ranks' tokens over the slowest rank's time
    assert res[0]["value"] == pytest.approx(8192 * 3 * 2 / 0.015)


def test_single_rank_needs_no_process_group():
    import bench
    rep = bench.Replicas(1, "cpu")
    rep.barrier()
    assert rep.max(12.5) == 12.5
    assert bench.job_throughput(100, 2, 1, 1000.0) == 200.0


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env["RANK"], env["LOCAL_RANK"] = "0", "0"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3", "--ref-step-seconds", "0.2"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
