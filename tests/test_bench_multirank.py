"""The benchmark's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Under torchrun each rank runs an independent replica (the forward needs no
exchange); the timing takes the slowest rank's time and the whole-job value
counts every rank's work.  These tests run the same helpers bench.py uses,
with a CPU tensor for the reduction, and check that the reference arm prints
only on rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist, cuda=False)
        my_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        worst = bench.max_over_ranks(dist, my_ms, device="cpu")
        value = bench.whole_job_tflops(1e12, 4, world, worst)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"worst": worst, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert res[0]["worst"] == res[1]["worst"] == 15.0
    # 2 ranks x 4 steps x 1 TFLOP in 15 ms
    assert res[0]["value"] == pytest.approx(2 * 4 * 1.0 / 0.015)


def test_whole_job_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_tflops(2e12, 10, 1, 20.0) == pytest.approx(1000.0)
    assert bench.max_over_ranks(None, 3.5) == 3.5


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_json_line():
    """The reference arm (the oracle on host cores) prints one JSON line with
    the contract's keys, on the same metric and workload as the GPU line."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"]["workload"] == bench.WORKLOAD and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
