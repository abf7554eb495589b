"""Decode Context Parallelism across GPUs: the exchange around the per-GPU call.

"Decode Context Parallelism" (section 4.1) runs each decode step as
AllGather Q -> Compute -> a combine of the partial outputs by their LSEs;
"Kimi K3 Performance Optimizations in vLLM" (section "Decode context
parallelism") does the output/LSE reduction with an all-to-all.  With one
process per GPU in a group of N ranks, rank r holding query heads
[r*H/N, (r+1)*H/N) and shard r of every request's latent cache (a *_local
layout: only its own positions, compactly), one step here is:

  1. all-gather of the query heads           -> q [B, q_len, H, 576] on every rank
  2. mla_decode_partial(shard_id = r)         -> this shard's (o, lse) for all H heads
  3. all-to-all of head slices of (o, lse)    -> every shard's partial of heads of rank r
  4. mla_shard_combine over the N partials    -> out [B, q_len, H/N, 512 | 128]
     (fused with W_UV of the rank's heads when given)

Steps 2 and 4 are the library's CUDA kernels; steps 1 and 3 are
torch.distributed collectives (NCCL on GPUs).  Per step a rank sends
(N-1)/N of its query heads (B*q_len*H/N*576*2 bytes to every peer) and of
its partials (B*q_len*H/N*(512+1)*4 bytes to every peer).  The result is
each rank's head slice, the layout a tensor-parallel output projection
takes next.

With chunks = k > 1 the requests are cut into k groups: the all-to-all of a
group's partials is started asynchronously (on NCCL's own stream on GPUs)
and the next group's partial attention runs meanwhile, so the exchange
overlaps compute; the combines follow once each exchange has landed.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

from . import DEFAULT_SCALE, mla_decode_partial, mla_shard_combine


def _world(group):
    import torch.distributed as dist
    if group is None and not (dist.is_available() and dist.is_initialized()):
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def gather_query_heads(q_local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of the query heads: [B, q_len, H/N, 576] per rank ->
    [B, q_len, H, 576], rank r's heads at [r*H/N, (r+1)*H/N)."""
    N, _ = _world(group)
    if N == 1:
        return q_local
    import torch.distributed as dist
    parts = [torch.empty_like(q_local) for _ in range(N)]
    dist.all_gather(parts, q_local.contiguous(), group=group)
    return torch.cat(parts, dim=2).contiguous()


class _HeadExchange:
    """An all-to-all of one partial's head slices, started at construction
    (asynchronously when there is a process group); wait() returns
    (partials [N, B, q_len, H/N, 512], lses [N, B, q_len, H/N])."""

    def __init__(self, o: torch.Tensor, lse: torch.Tensor, group=None):
        N, _ = _world(group)
        B, q_len, H, D = o.shape
        if H % N != 0:
            raise ValueError(f"{H} heads do not split over {N} ranks")
        Hl = H // N
        self.send_o = o.reshape(B, q_len, N, Hl, D).permute(2, 0, 1, 3, 4).contiguous()
        self.send_l = lse.reshape(B, q_len, N, Hl).permute(2, 0, 1, 3).contiguous()
        self.works = []
        if N == 1:
            self.recv_o, self.recv_l = self.send_o, self.send_l
            return
        import torch.distributed as dist
        self.recv_o = torch.empty_like(self.send_o)
        self.recv_l = torch.empty_like(self.send_l)
        self.works = [
            dist.all_to_all_single(self.recv_o, self.send_o, group=group, async_op=True),
            dist.all_to_all_single(self.recv_l, self.send_l, group=group, async_op=True),
        ]

    def wait(self):
        for w in self.works:
            w.wait()
        return self.recv_o, self.recv_l


def exchange_head_slices(o: torch.Tensor, lse: torch.Tensor, group=None):
    """All-to-all of this rank's partial (o [B, q_len, H, 512], lse
    [B, q_len, H]): rank k receives slice k of the heads from every shard.
    Returns (partials [N, B, q_len, H/N, 512], lses [N, B, q_len, H/N]),
    shard-major, the layout mla_shard_combine takes."""
    return _HeadExchange(o, lse, group).wait()


def _cuda_partial(q_full, kv, block_table, seq_lens, num_shards, layout, shard_id, kv_scale,
                  causal, softmax_scale, q_lens=None):
    o, lse, _ = mla_decode_partial(q_full, kv, block_table, seq_lens, num_shards,
                                   layout + "_local", shard_id=shard_id, kv_scale=kv_scale,
                                   causal=causal, softmax_scale=softmax_scale, q_lens=q_lens)
    return o[0], lse[0]


def _cuda_combine(partials, lses, w_uv, causal, softmax_scale):
    return mla_shard_combine(partials, lses, w_uv=w_uv, causal=causal,
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
    chunks: request groups whose exchange overlaps the next group's compute.
    Returns (out [B, q_len, H/N, 512 | 128] bf16, lse [B, q_len, H/N] fp32).

    partial_fn / combine_fn replace the library's CUDA calls (same arguments
    and results); the library's calls are the default.
    """
    N, rank = _world(group)
    partial_fn = partial_fn or _cuda_partial
    combine_fn = combine_fn or _cuda_combine
    q_full = gather_query_heads(q_local, group)
    B = q_full.shape[0]
    chunks = max(1, min(int(chunks), B))
    bounds = [B * c // chunks for c in range(chunks + 1)]
    exchanges = []
    for c in range(chunks):
        b0, b1 = bounds[c], bounds[c + 1]
        if b0 == b1:
            continue
        whole = b0 == 0 and b1 == B
        sub = (lambda t: t) if whole else (lambda t: t[b0:b1])
        o, lse = partial_fn(sub(q_full), kv, sub(block_table), sub(seq_lens), N, layout, rank,
                            kv_scale, causal, softmax_scale,
                            None if q_lens is None else sub(q_lens))
        exchanges.append(_HeadExchange(o, lse, group))   # runs while the next group computes
    outs, lses = [], []
    for ex in exchanges:
        partials, plse = ex.wait()
        out, lse = combine_fn(partials, plse, w_uv_local, causal, softmax_scale)
        outs.append(out)
        lses.append(lse)
    if len(outs) == 1:
        return outs[0], lses[0]
    return torch.cat(outs, 0), torch.cat(lses, 0)
