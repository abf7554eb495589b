"""The multi-GPU DCP exchange (query all-gather, head-sliced all-to-all of the
shard partials, LSE combine) on world-size 2 and 4 gloo ranks on CPU.

The CUDA compute calls are replaced on CPU by the oracle: rank r's partial is
the oracle's shard-r attention and the combine is the oracle's LSE merge and
W_UV projection.  What is under test is the exchange: the query each rank
computes with, which head slices travel where, and that every rank ends with
exactly its heads of unsharded attention -- also when the requests are cut
into groups whose exchanges run asynchronously behind the next group's
compute.
"""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload(layout, N, causal, wuv):
    lens = [1, 90, 700, 2500]
    return mi.build_workload("dcp", len(lens), 3 if causal else 1, 16 * N, lens, N, layout,
                             "bf16", causal, seed=500 + N, with_w_uv=wuv, poison=True)


def _worker(rank, world, port, layout, causal, wuv, chunks, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sequence_sharded_mla_gb300 import dcp
        w = _workload(layout, world, causal, wuv)
        B, q_len, H = w.batch, w.q_len, w.num_heads
        Hl = H // world
        q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16)
        q_local = q[:, :, rank * Hl:(rank + 1) * Hl].contiguous()
        local = mi.local_shard_cache(w, world, rank, layout, seed=rank)
        kv = torch.from_numpy(local["kv"].view(np.int16)).view(torch.bfloat16)
        bt = torch.from_numpy(local["block_table"])
        sl = torch.from_numpy(w.seq_lens)
        w_uv_local = None
        if wuv:
            w_uv_local = torch.from_numpy(w.w_uv.view(np.int16)).view(torch.bfloat16)[
                rank * Hl:(rank + 1) * Hl].contiguous()

        seen = {"q_ok": [], "groups": []}
        # the all-gathered query, rank-major: block k holds rank k's heads
        q_gathered = q.reshape(B, q_len, world, Hl, 576).permute(2, 0, 1, 3, 4)

        def partial_fn(q_g, b0, b1, kv_, bt_, sl_, N, lay, shard_id, kv_scale, causal_, scale,
                       q_lens=None):
            seen["q_ok"].append(torch.equal(q_g, q_gathered))
            seen["groups"].append((b0, b1))
            assert N == world and shard_id == rank and lay == layout and causal_ == causal
            assert kv_ is kv and bt_.storage_offset() == b0 * bt.shape[1]
            assert torch.equal(bt_, bt[b0:b1]) and torch.equal(sl_, sl[b0:b1])
            o, l = oracle.attend(w, shard=shard_id, num_shards=N, layout=lay)
            # head slices [N, b1 - b0, q_len, H/N, ...], slice k for rank k
            o = np.moveaxis(o.reshape(B, q_len, N, Hl, 512)[b0:b1], 2, 0)
            l = np.moveaxis(l.reshape(B, q_len, N, Hl)[b0:b1], 2, 0)
            return (torch.from_numpy(np.ascontiguousarray(o, dtype=np.float32)),
                    torch.from_numpy(np.ascontiguousarray(l, dtype=np.float32)))

        def combine_fn(partials, lses, w_uv, causal_, scale):
            n, bc = partials.shape[0], partials.shape[1]
            o, l = oracle.lse_merge(partials.double().numpy().reshape(n, -1, 512),
                                    lses.double().numpy().reshape(n, -1))
            l = torch.from_numpy(np.asarray(l)).reshape(bc, q_len, Hl)
            if w_uv is not None:
                heads = np.tile(np.arange(Hl, dtype=np.int32), bc * q_len)
                y = oracle.project_wuv(o, heads, w_uv.view(torch.int16).numpy().view(np.uint16))
                return torch.from_numpy(y).reshape(bc, q_len, Hl, 128), l
            return torch.from_numpy(o).reshape(bc, q_len, Hl, 512), l

        res, lse = dcp.dcp_decode_step(q_local, kv, bt, sl, layout=layout, causal=causal,
                                       w_uv_local=w_uv_local, partial_fn=partial_fn,
                                       combine_fn=combine_fn, chunks=chunks)
        groups = seen["groups"]
        assert len(groups) == min(chunks, B)
        assert groups[0][0] == 0 and groups[-1][1] == B
        assert all(a[1] == b[0] for a, b in zip(groups, groups[1:]))
        out[rank] = (all(seen["q_ok"]), res.numpy(), lse.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,layout,causal,wuv,chunks", [
    (2, "interleaved", False, False, 1),
    (2, "contiguous", True, True, 1),
    (4, "interleaved", True, False, 1),
    (4, "contiguous", False, True, 1),
    (2, "interleaved", True, True, 3),
    (4, "contiguous", False, False, 2),
])
def test_dcp_exchange_gives_each_rank_its_heads_of_unsharded_attention(world, layout, causal,
                                                                         wuv, chunks):
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), layout, causal, wuv, chunks, out),
                 nprocs=world, join=True)
        res = dict(out)
    w = _workload(layout, world, causal, wuv)
    ref, ref_lse, ref_y = oracle.reference_step(w)
    B, q_len, H = w.batch, w.q_len, w.num_heads
    Hl = H // world
    ref = (ref_y if wuv else ref).reshape(B, q_len, H, -1)
    ref_lse = ref_lse.reshape(B, q_len, H)
    for r in range(world):
        q_ok, got, lse = res[r]
        assert q_ok, f"rank {r} computed with a wrong query"
        sl = slice(r * Hl, (r + 1) * Hl)
        check_close(got.reshape(-1, got.shape[-1]), ref[:, :, sl].reshape(-1, ref.shape[-1]),
                    TOL_OUT, f"rank {r} out")
        check_close(lse.reshape(-1), ref_lse[:, :, sl].reshape(-1), TOL_LSE, f"rank {r} lse")


def test_head_slices_route_to_their_ranks_single_process():
    """Without a process group the exchange hands the one head slice back, and
    the query all-gather is the rank's own heads as a block of one."""
    from sequence_sharded_mla_gb300 import dcp
    o = torch.arange(1 * 2 * 1 * 32 * 512, dtype=torch.float32).reshape(1, 2, 1, 32, 512)
    lse = torch.arange(1 * 2 * 1 * 32, dtype=torch.float32).reshape(1, 2, 1, 32)
    po, pl = dcp.exchange_head_slices(o, lse)
    assert po.shape == (1, 2, 1, 32, 512) and torch.equal(po, o) and torch.equal(pl, lse)
    q = torch.randn(2, 1, 32, 576).to(torch.bfloat16)
    g = dcp.gather_query_heads(q)
    assert g.shape == (1, 2, 1, 32, 576) and torch.equal(g[0], q)
