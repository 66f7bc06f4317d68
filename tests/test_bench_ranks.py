"""The multi-GPU contract of bench.py, checked on CPU with gloo ranks: the
path shards as independent replicas (no collective on the data path), the
reported value is all ranks' units over the slowest rank's time, and under
torchrun only rank 0 prints the reference arm's JSON line."""
import json
import time
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    value, elapsed = bench.aggregate_over_ranks(1.0 + rank, 10.0, dist, "cpu")
    out[rank] = (value, elapsed)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_throughput_uses_max_time_and_all_units():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        value, elapsed = res[rank]
        assert elapsed == 2.0                 # slowest rank
        assert value == world * 10.0 / 2.0    # every rank's units over that time


def test_single_process_aggregate():
    import bench
    assert bench.aggregate_over_ranks(0.5, 100.0) == (200.0, 0.5)


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    t0 = time.perf_counter()
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=280)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # the line keeps the contract of the GPU arm's line: same keys, metric, unit and config
    import bench
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == "tok/s" and d["higher_is_better"] is True
    assert d["config"] == bench.workload_config("auto")
    assert d["n_gpus"] == 2 and d["steps"] == 1 and d["warmup"] == 0
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in d["cpu_baseline"], key
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    # a step is the bounded sample: its measured time fits inside the run's own wall clock,
    # and the scaled whole-step time is reported beside it
    assert 0 < d["ms_per_step"] / 1e3 <= wall
    assert d["extrapolated_ms_per_step"] >= d["ms_per_step"]
    assert abs(d["value"] - bench.B * bench.N / (d["extrapolated_ms_per_step"] / 1e3)) <= 1e-6 * d["value"]
