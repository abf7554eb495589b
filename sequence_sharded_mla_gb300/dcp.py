"""Decode Context Parallelism across GPUs: the exchange around the per-GPU call.

"Decode Context Parallelism" (section 4.1) runs each decode step as
AllGather Q -> Compute -> a combine of the partial outputs by their LSEs;
"Kimi K3 Performance Optimizations in vLLM" (section "Decode context
parallelism") does the output/LSE reduction with an all-to-all.  With one
process per GPU in a group of N ranks, rank r holding query heads
[r*H/N, (r+1)*H/N) and shard r of every request's latent cache (a *_local
layout: only its own positions, compactly), one step here is:

  1. all-gather of the query heads           -> [N, B, q_len, H/N, 576] on every rank
  2. mla_decode_partial_dcp(rank = r)         -> this shard's (o, lse) for all H heads,
                                                 written as N head slices
  3. all-to-all of the head slices            -> every shard's partial of heads of rank r
  4. mla_shard_combine over the N partials    -> out [B, q_len, H/N, 512 | 128]
     (fused with W_UV of the rank's heads when given)

Steps 2 and 4 are the library's CUDA kernels; steps 1 and 3 are
torch.distributed collectives (NCCL on GPUs).  Nothing is copied between
them: the partial kernel reads the query from the all-gather's rank-major
buffer and writes its outputs as the all-to-all's send buffers, and the
all-to-all lands them shard-major, as the combine takes them.  Per step a
rank sends (N-1)/N of its query heads (B*q_len*H/N*576*2 bytes to every
peer) and of its partials (B*q_len*H/N*(512+1)*4 bytes to every peer).  The
result is each rank's head slice, the layout a tensor-parallel output
projection takes next.

With chunks = k > 1 the requests are cut into k groups: the all-to-all of a
group's partials is started asynchronously (on NCCL's own stream on GPUs)
and the next group's partial attention runs meanwhile, so the exchange
overlaps compute; the combines follow once each exchange has landed, each
into its requests' rows of the output.  Every group is a launch of its own,
with its own start and tail (tens of microseconds on a GB300), so more than
one group pays only when the exchange takes longer than that.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

from . import D_UV, D_V, DEFAULT_SCALE, mla_decode_partial_dcp, mla_shard_combine


def _world(group):
    import torch.distributed as dist
    if group is None and not (dist.is_available() and dist.is_initialized()):
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def gather_query_heads(q_local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of the query heads: [B, q_len, H/N, 576] per rank ->
    [N, B, q_len, H/N, 576], rank r's block holding heads [r*H/N, (r+1)*H/N),
    the layout the collective lands (mla_decode_partial_dcp reads it as is)."""
    N, _ = _world(group)
    q_local = q_local.contiguous()
    if N == 1:
        return q_local.unsqueeze(0)
    import torch.distributed as dist
    out = torch.empty((N,) + tuple(q_local.shape), dtype=q_local.dtype, device=q_local.device)
    if dist.get_backend(group) == "gloo":
        dist.all_gather(list(out.unbind(0)), q_local, group=group)
    else:
        dist.all_gather_into_tensor(out, q_local, group=group)
    return out


class _HeadExchange:
    """An all-to-all of one partial's head slices, started at construction
    (asynchronously when there is a process group).  send_o [N, B, q_len,
    H/N, 512] and send_l [N, B, q_len, H/N] hold slice k for rank k; wait()
    returns what every rank sent this one: (partials [N, B, q_len, H/N, 512],
    lses [N, B, q_len, H/N]), shard-major."""

    def __init__(self, send_o: torch.Tensor, send_l: torch.Tensor, group=None):
        N, _ = _world(group)
        if send_o.shape[0] != N or send_l.shape[0] != N:
            raise ValueError(f"send buffers must hold {N} head slices")
        self.works = []
        if N == 1:
            self.recv_o, self.recv_l = send_o, send_l
            return
        import torch.distributed as dist
        self.recv_o = torch.empty_like(send_o)
        self.recv_l = torch.empty_like(send_l)
        self.works = [
            dist.all_to_all_single(self.recv_o, send_o, group=group, async_op=True),
            dist.all_to_all_single(self.recv_l, send_l, group=group, async_op=True),
        ]

    def wait(self):
        for w in self.works:
            w.wait()
        return self.recv_o, self.recv_l


def exchange_head_slices(send_o: torch.Tensor, send_l: torch.Tensor, group=None):
    """All-to-all of this rank's partial in head slices (send_o [N, B, q_len,
    H/N, 512], send_l [N, B, q_len, H/N], slice k for rank k): returns
    (partials [N, B, q_len, H/N, 512], lses [N, B, q_len, H/N]), shard-major,
    the layout mla_shard_combine takes."""
    return _HeadExchange(send_o, send_l, group).wait()


def _cuda_partial(q_gathered, b0, b1, kv, block_table, seq_lens, num_shards, layout, shard_id,
                  kv_scale, causal, softmax_scale, q_lens=None):
    o, lse, _ = mla_decode_partial_dcp(q_gathered, kv, block_table, seq_lens, shard_id,
                                       layout + "_local", batch_first=b0, kv_scale=kv_scale,
                                       causal=causal, softmax_scale=softmax_scale, q_lens=q_lens)
    return o, lse


def _cuda_combine(partials, lses, w_uv, causal, softmax_scale, out=None, lse_out=None):
    return mla_shard_combine(partials, lses, w_uv=w_uv, out=out, lse_out=lse_out, causal=causal,
                             softmax_scale=softmax_scale)


def dcp_decode_step(q_local: torch.Tensor, kv: torch.Tensor, block_table: torch.Tensor,
                    seq_lens: torch.Tensor, *, group=None, layout: str = "interleaved",
                    kv_scale: Optional[torch.Tensor] = None, causal: bool = False,
                    softmax_scale: float = DEFAULT_SCALE, w_uv_local: Optional[torch.Tensor] = None,
                    q_lens: Optional[torch.Tensor] = None, partial_fn: Optional[Callable] = None,
                    combine_fn: Optional[Callable] = None, chunks: int = 1):
    """One sharded decode step of attention on this rank.

    q_local: bf16 [B, q_len, H/N, 576], this rank's query heads.
    kv, block_table (and kv_scale for fp8): this rank's local slice of the
    latent cache (shard `rank` of N under `layout`, stored compactly: see
    mla_layout's *_LOCAL layouts).  seq_lens: the global lengths [B].
    w_uv_local: bf16 [H/N, 512, 128], W_UV of this rank's heads, or None.
    q_lens: optional int32 [B] query tokens per request of a padded batch.
    chunks: request groups whose exchange overlaps the next group's compute
    (1, the default: one launch over the whole batch).
    Returns (out [B, q_len, H/N, 512 | 128] bf16, lse [B, q_len, H/N] fp32).

    partial_fn / combine_fn replace the library's CUDA calls; the library's
    calls are the default.  partial_fn(q_gathered [N, B, q_len, H/N, 576], b0,
    b1, kv, block_table[b0:b1], seq_lens[b0:b1], N, layout, rank, kv_scale,
    causal, softmax_scale, q_lens[b0:b1] or None) returns this shard's partial
    of requests b0..b1-1 as head slices: (o [N, b1-b0, q_len, H/N, 512], lse
    [N, b1-b0, q_len, H/N]), slice k for rank k.  combine_fn(partials, lses,
    w_uv_local, causal, softmax_scale) returns (out, lse) of those requests.
    """
    N, rank = _world(group)
    default_combine = combine_fn is None
    partial_fn = partial_fn or _cuda_partial
    combine_fn = combine_fn or _cuda_combine
    q_g = gather_query_heads(q_local, group)
    B = q_g.shape[1]
    chunks = max(1, min(int(chunks), B))
    bounds = [B * c // chunks for c in range(chunks + 1)]
    groups = []
    for c in range(chunks):
        b0, b1 = bounds[c], bounds[c + 1]
        if b0 == b1:
            continue
        whole = b0 == 0 and b1 == B
        sub = (lambda t: t) if whole else (lambda t: t[b0:b1])
        o, lse = partial_fn(q_g, b0, b1, kv, sub(block_table), sub(seq_lens), N, layout, rank,
                            kv_scale, causal, softmax_scale,
                            None if q_lens is None else sub(q_lens))
        groups.append((b0, b1, _HeadExchange(o, lse, group)))   # runs while the next group computes
    if len(groups) == 1:
        partials, plse = groups[0][2].wait()
        return combine_fn(partials, plse, w_uv_local, causal, softmax_scale)
    if default_combine:
        # each group's combine writes its requests' rows of the output
        q_len, Hl = q_g.shape[2], q_g.shape[3]
        d = D_V if w_uv_local is None else D_UV
        out = torch.empty((B, q_len, Hl, d), dtype=torch.bfloat16, device=q_g.device)
        lse_out = torch.empty((B, q_len, Hl), dtype=torch.float32, device=q_g.device)
        for b0, b1, ex in groups:
            partials, plse = ex.wait()
            _cuda_combine(partials, plse, w_uv_local, causal, softmax_scale,
                          out=out[b0:b1], lse_out=lse_out[b0:b1])
        return out, lse_out
    outs, lses = [], []
    for _, _, ex in groups:
        partials, plse = ex.wait()
        o, l = combine_fn(partials, plse, w_uv_local, causal, softmax_scale)
        outs.append(o)
        lses.append(l)
    return torch.cat(outs, 0), torch.cat(lses, 0)
