"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The prefill shards with no exchange (independent heads and decode states), so
the only cross-rank steps are the timing ones: a barrier on both sides of the
timed region and the maximum of the per-rank times, from which rank 0 reports
the whole-job rate.  These tests run those steps in two real processes, and
the reference arm under torchrun (rank 0 alone works and prints one line; the
other rank exits 0 without work).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, _, dist = bench.dist_setup()
    assert (r, w) == (rank, world) and dist is not None
    bench.barrier(dist, torch)
    mx = bench.max_over_ranks(1.5 + rank, dist)           # per-rank "times" 1.5 and 2.5
    mn = -bench.max_over_ranks(-(1.5 + rank), dist)       # the same reduction, negated
    bench.barrier(dist, torch)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": mx, "min": mn, "backend": dist.get_backend()}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["backend"] == "gloo"
        assert r["max"] == 2.5 and r["min"] == 1.5  # every rank sees the slowest rank's time


def test_reference_arm_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", f"--master-port={port}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--ref-tokens", "128"]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_line_carries_the_contract_keys():
    """One process, no GPU: the reference arm's JSON line has every key of the
    bench contract, its e2e value equals its own value with no copies, and its
    cpu_baseline describes the same run."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--ref-tokens", "64"]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and "workload" in d["config"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
