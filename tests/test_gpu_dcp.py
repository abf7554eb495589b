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
    # the query all-gather as it lands: rank-major blocks of H/N heads
    q_g = q.reshape(B, q_len, N, Hl, 576).permute(2, 0, 1, 3, 4).contiguous()
    sl = torch.from_numpy(w.seq_lens).to(dev)
    outs, lses = [], []
    for s in range(N):
        d = mi.local_shard_cache(w, N, s, layout, seed=s)
        kv = torch.from_numpy(d["kv"].view(np.int16)).view(torch.bfloat16).to(dev)
        bt = torch.from_numpy(d["block_table"]).to(dev)
        o, l = dcp._cuda_partial(q_g, 0, B, kv, bt, sl, N, layout, s, None, False,
                                 w.softmax_scale)
        outs.append(o)        # [N, B, q_len, H/N, 512]: slice r for rank r
        lses.append(l)
    wuv_t = None
    if wuv:
        wuv_t = torch.from_numpy(w.w_uv.view(np.int16)).view(torch.bfloat16).to(dev)
    ref, ref_lse, ref_y = oracle.reference_step(w)
    ref = (ref_y if wuv else ref).reshape(B, q_len, H, -1)
    ref_lse = ref_lse.reshape(B, q_len, H)
    for r in range(N):
        hs = slice(r * Hl, (r + 1) * Hl)
        # the all-to-all: rank r receives slice r of every shard's partial
        partials = torch.stack([o[r] for o in outs]).contiguous()
        plse = torch.stack([l[r] for l in lses]).contiguous()
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


@pytest.mark.parametrize("N,layout,kv_dtype,q_len,causal,H,q_lens,groups", [
    (2, "interleaved", "bf16", 1, False, 64, None, 1),
    (4, "contiguous", "bf16", 3, True, 64, [1, 3, 2, 3], 2),
    (8, "interleaved", "bf16", 2, True, 64, None, 3),
    (2, "interleaved", "fp8", 1, False, 64, None, 2),
    (4, "interleaved", "fp8", 9, True, 64, [9, 4, 1, 7], 1),
    (2, "contiguous", "bf16", 1, False, 128, None, 1),
    (1, "interleaved", "bf16", 2, True, 128, None, 2),
])
def test_rank_major_io_matches_the_oracle(N, layout, kv_dtype, q_len, causal, H, q_lens, groups):
    """mla_decode_partial_dcp reads the query from the all-gather's rank-major
    buffer and writes its partial as the all-to-all's send buffers; every
    element of them against the oracle's shard partial, for request groups
    that start inside the gathered batch, units split across CTAs (long
    contexts, whose pieces the merge writes) and padding rows."""
    import torch
    import sequence_sharded_mla_gb300 as mla
    dev = torch.device("cuda:0")
    lens = [20000, 3, 777, 9000]
    fp8 = kv_dtype == "fp8"
    w = mi.build_workload("dcp-io", len(lens), q_len, H, lens, N, layout, kv_dtype, causal,
                          seed=700 + N + q_len, kv_sigma=1.0 if fp8 else 0.5, poison=True,
                          q_lens=q_lens)
    B, Hl = w.batch, H // N
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(dev)
    q_g = q.reshape(B, q_len, N, Hl, 576).permute(2, 0, 1, 3, 4).contiguous()
    sl = torch.from_numpy(w.seq_lens).to(dev)
    ql = None if q_lens is None else torch.from_numpy(w.q_lens).to(dev)
    bounds = [B * c // groups for c in range(groups + 1)]
    for s in range(N):
        d = mi.local_shard_cache(w, N, s, layout, seed=s)
        if fp8:
            kv = torch.from_numpy(d["kv"]).to(dev)
            sc = torch.from_numpy(d["kv_scale"]).to(dev)
        else:
            kv = torch.from_numpy(d["kv"].view(np.int16)).view(torch.bfloat16).to(dev)
            sc = None
        bt = torch.from_numpy(d["block_table"]).to(dev)
        ro, rl = oracle.attend(w, shard=s, num_shards=N, layout=layout)
        ro = ro.reshape(B, q_len, N, Hl, 512)
        rl = rl.reshape(B, q_len, N, Hl)
        for b0, b1 in zip(bounds, bounds[1:]):
            o, l, ws = mla.mla_decode_partial_dcp(
                q_g, kv, bt[b0:b1], sl[b0:b1], s, layout + "_local", batch_first=b0,
                kv_scale=sc, causal=causal, softmax_scale=w.softmax_scale,
                q_lens=None if ql is None else ql[b0:b1])
            torch.cuda.synchronize()
            assert mla.mla_get_device_error(ws) == 0
            assert o.shape == (N, b1 - b0, q_len, Hl, 512)
            want_o = np.moveaxis(ro[b0:b1], 2, 0)
            want_l = np.moveaxis(rl[b0:b1], 2, 0)
            check_close(o.cpu().numpy().reshape(-1, 512), want_o.reshape(-1, 512), TOL_OUT,
                        f"shard {s} requests {b0}..{b1}", rel=REL_OUT)
            check_close(l.cpu().numpy().reshape(-1), want_l.reshape(-1), TOL_LSE,
                        f"shard {s} lse {b0}..{b1}")
