"""Host logic of the multi-GPU benchmark, on CPU: world-size-2 gloo ranks.

With N GPUs every rank decodes its own, independently seeded batch of the
same shape (weak scaling, no data-path collective); the job's time is the
slowest rank's and its work the sum over ranks.  Under torchrun the
reference arm runs on rank 0 alone and prints one line.
"""
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
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [1.0 + rank, 10.0 * (world - rank), 0.5]
        res = bench.reduce_over_ranks(dist, times, 100 * (rank + 1), torch.device("cpu"))
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_takes_max_time_and_total_bytes():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_reduce_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        times, total = res[r]
        assert times == [2.0, 20.0, 0.5]
        assert total == 300.0


def test_single_rank_reduction_is_identity():
    times, total = bench.reduce_over_ranks(None, [3.0, 4.0], 12345, torch.device("cpu"))
    assert times == [3.0, 4.0] and total == 12345.0


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5])
def test_rank_workloads_are_independent_batches_of_one_shape(config):
    base = bench.rank_workload_params(config, 0)
    seeds = set()
    for rank in range(8):
        p = bench.rank_workload_params(config, rank)
        for k in ("batch", "q_len", "num_heads", "num_shards", "layout", "kv_dtype", "causal"):
            assert p[k] == base[k], (rank, k)
        assert len(p["seq_lens"]) == p["batch"]
        seeds.add(p["seed"])
        if config == 2:
            assert int(np.sum(p["seq_lens"])) <= 4 * 1024 * 1024
            if rank > 0:
                assert list(p["seq_lens"]) != list(base["seq_lens"])
    assert len(seeds) == 8


def test_profiling_subset_keeps_first_requests():
    p = bench.rank_workload_params(2, 0, requests=4)
    full = bench.rank_workload_params(2, 0)
    assert p["batch"] == 4 and list(p["seq_lens"]) == list(full["seq_lens"])[:4]


def test_clock_sample_summary():
    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2055, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage"]
    res = bench.parse_clock_samples(rows)
    assert res == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--config", "1",
           "--ref-step-seconds", "0.05"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
