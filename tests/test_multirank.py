"""The multi-GPU path of the benchmark (replicas, no data-path collective) on the host:
two gloo ranks on CPU exercise the per-rank seed, the barrier and max-over-ranks timing
reduction and the whole-job throughput; the reference arm prints on rank 0 only."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = load_bench()
    import moe_inputs as mi
    cfg = mi.CONFIGS["tiny"]
    seed = bench.replica_seed(rank)
    x, _ = mi.activations(cfg, seed)
    local_ms = [12.5, 20.0][rank]  # the second rank is the slower one
    dist.barrier()
    total = bench.max_over_ranks(local_ms, world, "cpu")
    value = bench.job_throughput(world, cfg.T, 10, total)
    np.save(os.path.join(out_dir, "x%d.npy" % rank), x)
    with open(os.path.join(out_dir, "r%d.json" % rank), "w") as f:
        json.dump({"seed": seed, "total": total, "value": value}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r = [json.load(open(tmp_path / ("r%d.json" % i))) for i in range(world)]
    assert [q["seed"] for q in r] == [0, 1]
    assert r[0]["total"] == r[1]["total"] == 20.0           # the slowest rank's time on every rank
    assert r[0]["value"] == pytest.approx(2 * 16 * 10 / 20e-3)  # both ranks' tokens over that time
    x0, x1 = np.load(tmp_path / "x0.npy"), np.load(tmp_path / "x1.npy")
    assert x0.shape == x1.shape and not np.array_equal(x0, x1)  # each replica its own batch


def test_single_rank_needs_no_process_group():
    bench = load_bench()
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(1, 32, 200, 100.0) == pytest.approx(64000.0)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
