"""bench.py's multi-GPU DCP mode, its host logic on two gloo ranks on CPU.

run_dcp gives rank r its query heads and the cache slice of shard r, times
the DCP step (query all-gather, partial, head-sliced all-to-all, combine) and
assembles the JSON line.  Here the two CUDA calls are replaced by the oracle
(rank r's partial is the oracle's shard-r attention, the combine its LSE
merge), so what is under test is the bench's own part: the inputs each rank
gets, that the step it times returns each rank's heads of unsharded
attention, the exchange byte counts and the fields of the line.
"""
import argparse
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import mla_inputs as mi
import oracle
from _helpers import TOL_LSE, TOL_OUT, check_close

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    return mi.build_workload("benchdcp", 3, 1, 32, [90, 700, 1500], 2, "interleaved", "bf16",
                             False, seed=800, poison=True)


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w = _workload()
        B, q_len, H = w.batch, w.q_len, w.num_heads
        Hl = H // world
        calls = {"partial": 0, "outs": []}

        def partial_fn(q_g, b0, b1, kv_, bt_, sl_, N, lay, shard_id, kv_scale, causal_, scale,
                       q_lens=None):
            calls["partial"] += 1
            assert N == world and shard_id == rank and lay == "interleaved"
            assert sl_.storage_offset() == b0 and sl_.shape[0] == b1 - b0
            q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16)
            # the all-gathered query, rank-major: block k holds rank k's heads
            assert torch.equal(q_g, q.reshape(B, q_len, N, Hl, 576).permute(2, 0, 1, 3, 4))
            o, l = oracle.attend(w, shard=shard_id, num_shards=N, layout=lay)
            o = np.moveaxis(o.reshape(B, q_len, N, Hl, 512)[b0:b1], 2, 0)
            l = np.moveaxis(l.reshape(B, q_len, N, Hl)[b0:b1], 2, 0)
            return (torch.from_numpy(np.ascontiguousarray(o, dtype=np.float32)),
                    torch.from_numpy(np.ascontiguousarray(l, dtype=np.float32)))

        def combine_fn(partials, lses, w_uv, causal_, scale):
            n, bc = partials.shape[0], partials.shape[1]
            o, l = oracle.lse_merge(partials.double().numpy().reshape(n, -1, 512),
                                    lses.double().numpy().reshape(n, -1))
            res = (torch.from_numpy(o).reshape(bc, q_len, Hl, 512),
                   torch.from_numpy(np.asarray(l)).reshape(bc, q_len, Hl))
            calls["outs"].append(res)
            return res

        args = argparse.Namespace(config=2, requests=0, layout="", warmup=1, steps=2,
                                  dcp_chunks=2)
        line = bench.run_dcp(args, world, rank, dist, torch.device("cpu"), workload=w,
                             partial_fn=partial_fn, combine_fn=combine_fn)
        inp = bench.dcp_rank_inputs(w, world, rank, torch.device("cpu"))
        last = calls["outs"][-2:]                     # the last step's two request groups
        out[rank] = dict(line=line, partial_calls=calls["partial"],
                         out=torch.cat([o for o, _ in last], 0).numpy(),
                         lse=torch.cat([l for _, l in last], 0).numpy(),
                         q_local=inp["q_local"].view(torch.int16).numpy(),
                         local_tokens=inp["local_tokens"])
    finally:
        dist.destroy_process_group()


def test_bench_dcp_mode_on_two_gloo_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    w = _workload()
    B, q_len, H = w.batch, w.q_len, w.num_heads
    Hl = H // world
    ref, ref_lse, _ = oracle.reference_step(w)
    ref = ref.reshape(B, q_len, H, 512)
    ref_lse = ref_lse.reshape(B, q_len, H)
    for r in range(world):
        got = res[r]
        # warm-up 1 + 2 timed steps, two request groups each
        assert got["partial_calls"] == 3 * 2
        hs = slice(r * Hl, (r + 1) * Hl)
        assert np.array_equal(got["q_local"], w.q[:, :, hs].view(np.int16))
        check_close(got["out"].reshape(-1, 512), ref[:, :, hs].reshape(-1, 512), TOL_OUT,
                    f"rank {r} out")
        check_close(got["lse"].reshape(-1), ref_lse[:, :, hs].reshape(-1), TOL_LSE,
                    f"rank {r} lse")
    # every token is in exactly one rank's slice
    assert res[0]["local_tokens"] + res[1]["local_tokens"] == w.total_tokens
    line = res[0]["line"]
    assert res[1]["line"] is None
    assert line["n_gpus"] == 2 and line["scaling"] == "strong" and line["steps"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["config"]["num_shards"] == 2
    assert line["config"]["total_kv_bytes"] == w.kv_bytes()
    rows_l = B * q_len * Hl
    ex = line["exchange"]
    assert ex["q_allgather_bytes_per_rank"] == rows_l * 576 * 2
    assert ex["partial_alltoall_bytes_per_rank"] == rows_l * 513 * 4
    assert ex["chunks"] == 2
