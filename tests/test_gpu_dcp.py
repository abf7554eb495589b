"""The per-rank calls of the multi-GPU DCP step on one GPU: every rank's
CUDA partial over its local cache slice, the head-slice exchange emulated by
slicing, and each rank's CUDA combine (fused with its W_UV) against the
oracle.  The collectives themselves are covered by the gloo tests."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from _helpers import REL_OUT, TOL_LSE, TOL_OUT, bf16_to_np, check_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,layout,wuv", [(1, "interleaved", False), (2, "interleaved", True),
                                          (4, "contiguous", False), (8, "interleaved", True)])
def test_rank_calls_of_a_dcp_step(N, layout, wuv):
    import torch
    from sequence_sharded_mla_gb300 import dcp
    dev = torch.device("cuda:0")
    lens = [3, 500, 2100, 6000]
    H = 64
    w = mi.build_workload("dcp-gpu", len(lens), 1, H, lens, N, layout, "bf16", False,
                          seed=600 + N, with_w_uv=wuv, poison=True)
    B, q_len = w.batch, w.q_len
    Hl = H // N
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    outs, lses = [], []
    for s in range(N):
        d = mi.local_shard_cache(w, N, s, layout, seed=s)
        kv = torch.from_numpy(d["kv"].view(np.int16)).view(torch.bfloat16).to(dev)
        bt = torch.from_numpy(d["block_table"]).to(dev)
        o, l = dcp._cuda_partial(q, kv, bt, sl, N, layout, s, None, False, w.softmax_scale)
        outs.append(o)
        lses.append(l)
    wuv_t = None
    if wuv:
        wuv_t = torch.from_numpy(w.w_uv.view(np.int16)).view(torch.bfloat16).to(dev)
    ref, ref_lse, ref_y = oracle.reference_step(w)
    ref = (ref_y if wuv else ref).reshape(B, q_len, H, -1)
    ref_lse = ref_lse.reshape(B, q_len, H)
    for r in range(N):
        hs = slice(r * Hl, (r + 1) * Hl)
        partials = torch.stack([o[:, :, hs] for o in outs]).contiguous()
        plse = torch.stack([l[:, :, hs] for l in lses]).contiguous()
        out, lse = dcp._cuda_combine(partials, plse,
                                     None if wuv_t is None else wuv_t[hs].contiguous(), False,
                                     w.softmax_scale)
        torch.cuda.synchronize()
        check_close(bf16_to_np(out).reshape(-1, out.shape[-1]),
                    ref[:, :, hs].reshape(-1, ref.shape[-1]), TOL_OUT, f"rank {r}", rel=REL_OUT)
        check_close(lse.cpu().numpy().reshape(-1), ref_lse[:, :, hs].reshape(-1), TOL_LSE,
                    f"rank {r} lse")


@pytest.mark.parametrize("chunks", [1, 2, 3])
def test_single_rank_step_without_a_process_group(chunks):
    """chunks > 1: the requests are run in groups (the CUDA partial on a slice
    of the block table and lengths), which must not change the result."""
    import torch
    from sequence_sharded_mla_gb300 import dcp
    dev = torch.device("cuda:0")
    w = mi.build_workload("dcp-1", 3, 1, 32, [77, 3000, 640], 1, "interleaved", "bf16", False,
                          seed=650)
    d = mi.local_shard_cache(w, 1, 0, "interleaved")
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(dev)
    kv = torch.from_numpy(d["kv"].view(np.int16)).view(torch.bfloat16).to(dev)
    out, lse = dcp.dcp_decode_step(q, kv, torch.from_numpy(d["block_table"]).to(dev),
                                   torch.from_numpy(w.seq_lens).to(dev), chunks=chunks)
    torch.cuda.synchronize()
    ref, ref_lse, _ = oracle.reference_step(w)
    check_close(bf16_to_np(out).reshape(-1, 512), ref, TOL_OUT, "out", rel=REL_OUT)
    check_close(lse.cpu().numpy().reshape(-1), ref_lse, TOL_LSE, "lse")
