"""Seeded synthetic workloads for sharded MLA decode.

This module only *makes inputs*: query rows, a paged latent cache (bf16, or
fp8 e4m3 with one fp32 scale per token), a block table, per-request context
lengths and the per-head value up-projection.  It performs none of the
attention arithmetic; the fp64 oracle and the CUDA path both read the bytes
produced here.

Workload recipes follow the five configurations of the benchmark suite
(MLA latent dims: 512 c_kv + 64 k_rope = 576, V = c_kv, page size 64,
softmax scale 1/sqrt(192)).  The agentic-trace length mix is a synthetic
stand-in for the trace described in "Decode Context Parallelism" section 2.1
(median ~67k, ~47% under 64k, ~18% under 8k, ~8% over 128k, ~3-4% over 256k,
tail up to ~1M).
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import build as _build

D_QK = 576          # 512 latent (c_kv) + 64 rope
D_V = 512           # V = c_kv
D_ROPE = 64
PAGE = 64
D_UV = 128          # per-head value up-projection output width
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)

# stream ids of the counter-based generator
S_Q, S_KV, S_PERM, S_LEN, S_WUV = 1, 2, 3, 4, 5

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u64, sz, dbl, vp = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_double, ctypes.c_void_p
        L.gen_normal_bf16.argtypes = [u64, u64, u64, sz, dbl, vp]
        L.gen_normal_f32.argtypes = [u64, u64, u64, sz, dbl, vp]
        L.gen_normal_fp8_rows.argtypes = [u64, u64, u64, sz, ctypes.c_int, dbl, vp, vp]
        L.quantize_fp8_rows.argtypes = [vp, sz, ctypes.c_int, vp, vp]
        L.encode_e4m3.argtypes = [vp, sz, vp]
        L.gen_u64.argtypes = [u64, u64, sz, vp]
        L.gen_permutation.argtypes = [u64, u64, sz, vp]
        L.fill_rows_u16.argtypes = [vp, vp, sz, ctypes.c_int, ctypes.c_uint16]
        L.fill_rows_u8.argtypes = [vp, vp, sz, ctypes.c_int, ctypes.c_uint8]
        for f in ("gen_normal_bf16", "gen_normal_f32", "gen_normal_fp8_rows",
                  "quantize_fp8_rows", "encode_e4m3", "gen_u64", "gen_permutation",
                  "fill_rows_u16", "fill_rows_u8"):
            getattr(L, f).restype = None
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return ctypes.c_void_p(a.ctypes.data)


# ----------------------------------------------------------------- primitives
def normal_bf16(seed, sid, shape, sigma, out=None, offset=0):
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    lib().gen_normal_bf16(seed, sid, offset, n, float(sigma), _ptr(out))
    return out


def normal_f32(seed, sid, shape, sigma, offset=0):
    out = np.empty(shape, dtype=np.float32)
    lib().gen_normal_f32(seed, sid, offset, int(np.prod(shape)), float(sigma), _ptr(out))
    return out


def normal_fp8_rows(seed, sid, nrows, width, sigma, codes=None, scales=None):
    if codes is None:
        codes = np.empty((nrows, width), dtype=np.uint8)
    if scales is None:
        scales = np.empty((nrows,), dtype=np.float32)
    lib().gen_normal_fp8_rows(seed, sid, 0, nrows, width, float(sigma), _ptr(codes), _ptr(scales))
    return codes, scales


def quantize_fp8_rows(x: np.ndarray):
    x = np.ascontiguousarray(x, dtype=np.float32)
    nrows, width = x.reshape(-1, x.shape[-1]).shape
    codes = np.empty((nrows, width), dtype=np.uint8)
    scales = np.empty((nrows,), dtype=np.float32)
    lib().quantize_fp8_rows(_ptr(x), nrows, width, _ptr(codes), _ptr(scales))
    return codes, scales


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(x.shape, dtype=np.uint8)
    lib().encode_e4m3(_ptr(x), x.size, _ptr(out))
    return out


def u64(seed, sid, n):
    out = np.empty((n,), dtype=np.uint64)
    lib().gen_u64(seed, sid, n, _ptr(out))
    return out


def uniform01(seed, sid, n):
    return (u64(seed, sid, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def permutation(seed, sid, n):
    out = np.empty((n,), dtype=np.int32)
    lib().gen_permutation(seed, sid, n, _ptr(out))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even); returns the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, np.uint16(0x7FC0), r)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------- length mixes
def agentic_lengths(seed: int, batch: int = 32, cap_total: int = 4 * 1024 * 1024):
    """Stratified piecewise log-uniform context lengths for the bimodal batch.

    Band counts for batch 32 reproduce the trace shape: 15 short (6 below 8k,
    9 in [8k,64k)), 17 long (2 in [64k, 67k) so the median lands near 67k,
    12 in [67k,128k), 2 in [128k,256k), 1 in [256k,1M]).  Each length is
    log-uniform inside its band; the batch order is then shuffled.  If the
    total exceeds ``cap_total`` the longest request is clamped.
    """
    bands = [(1024, 8192, 6), (8192, 65536, 9), (65536, 68608, 2),
             (68608, 131072, 12), (131072, 262144, 2), (262144, 1048577, 1)]
    counts = [c for _, _, c in bands]
    assert sum(counts) == 32
    scale = batch / 32.0
    u = uniform01(seed, S_LEN, 4 * batch + 64)
    lens, k = [], 0
    for lo, hi, c in bands:
        n = max(1, int(round(c * scale))) if batch != 32 else c
        for _ in range(n):
            v = math.exp(math.log(lo) + u[k] * (math.log(hi) - math.log(lo)))
            lens.append(min(max(int(v), lo), hi - 1))
            k += 1
    lens = lens[:batch]
    while len(lens) < batch:
        lens.append(8192)
    perm = permutation(seed, S_LEN + 100, len(lens))
    lens = [lens[i] for i in perm]
    tot = sum(lens)
    if tot > cap_total:
        i = int(np.argmax(lens))
        lens[i] -= tot - cap_total
    return np.array(lens, dtype=np.int32)


def uniform_lengths(seed: int, batch: int, lo: int, hi: int):
    x = u64(seed, S_LEN, batch) >> np.uint64(32)
    span = np.uint64(hi - lo + 1)
    return (np.uint64(lo) + ((x * span) >> np.uint64(32))).astype(np.int32)


# ---------------------------------------------------------------- workload
@dataclass
class Workload:
    name: str
    batch: int
    q_len: int
    num_heads: int
    seq_lens: np.ndarray               # int32 [B]
    num_shards: int
    layout: str                        # "interleaved" | "contiguous"
    kv_dtype: str                      # "bf16" | "fp8"
    causal: bool
    seed: int
    q: np.ndarray = None               # uint16 (bf16 bits) [B, q_len, H, 576]
    kv: np.ndarray = None              # uint16 [P, 64, 576] or uint8 [P, 64, 576]
    kv_scale: Optional[np.ndarray] = None  # float32 [P, 64] (fp8 only)
    block_table: np.ndarray = None     # int32 [B, max_pages]
    w_uv: Optional[np.ndarray] = None  # uint16 [H, 512, 128] or None
    q_lens: Optional[np.ndarray] = None  # int32 [B]: query tokens per request (None: all q_len)
    softmax_scale: float = SOFTMAX_SCALE
    notes: dict = field(default_factory=dict)

    @property
    def num_pages(self):
        return self.kv.shape[0]

    @property
    def max_pages(self):
        return self.block_table.shape[1]

    @property
    def total_tokens(self):
        return int(np.sum(self.seq_lens.astype(np.int64)))

    def kv_bytes(self):
        """Algorithmic KV bytes one full pass reads: every token < L_b once
        (576 bf16 = 1152 B, or 576 e4m3 codes + a 4-byte scale = 580 B)."""
        per = 1152 if self.kv_dtype == "bf16" else 580
        return self.total_tokens * per


def build_workload(name, batch, q_len, num_heads, seq_lens, num_shards, layout,
                   kv_dtype, causal, seed, q_sigma=0.5, kv_sigma=0.5,
                   with_w_uv=False, w_sigma=0.02, extra_pages=0, poison=False,
                   pinned=False, max_pages=None, q_lens=None):
    """Generate every tensor of one workload.

    Pages are assigned to requests through a seeded random permutation of the
    whole pool, so each request's pages are scattered.  ``poison`` fills the
    rows past each request's end and all unreferenced pages with NaN (bf16
    0x7FC0, e4m3 0x7F, scale NaN) so that any read of them shows up.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (batch,)
    pages_per = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    used = int(pages_per.sum())
    P = used + extra_pages
    mp = int(pages_per.max()) if max_pages is None else max_pages
    mp = max(mp, 1)
    perm = permutation(seed, S_PERM, P)
    bt = np.full((batch, mp), -1, dtype=np.int32)
    off = 0
    for b in range(batch):
        n = int(pages_per[b])
        bt[b, :n] = perm[off:off + n]
        off += n

    def alloc(shape, dtype):
        if pinned:
            import torch
            tdt = {np.uint16: torch.int16, np.uint8: torch.uint8, np.float32: torch.float32}[dtype]
            t = torch.empty(shape, dtype=tdt, pin_memory=True)
            return t.numpy().view(dtype)
        return np.empty(shape, dtype=dtype)

    q = alloc((batch, q_len, num_heads, D_QK), np.uint16)
    normal_bf16(seed, S_Q, q.shape, q_sigma, out=q)
    kv_scale = None
    if kv_dtype == "bf16":
        kv = alloc((P, PAGE, D_QK), np.uint16)
        normal_bf16(seed, S_KV, kv.shape, kv_sigma, out=kv)
    elif kv_dtype == "fp8":
        kv = alloc((P, PAGE, D_QK), np.uint8)
        kv_scale = alloc((P, PAGE), np.float32)
        normal_fp8_rows(seed, S_KV, P * PAGE, D_QK, kv_sigma,
                        codes=kv.reshape(P * PAGE, D_QK), scales=kv_scale.reshape(-1))
    else:
        raise ValueError(kv_dtype)
    if poison:
        flag = np.ones((P, PAGE), dtype=np.uint8)
        for b in range(batch):
            L = int(seq_lens[b])
            for k in range(int(pages_per[b])):
                pg = bt[b, k]
                rows = min(PAGE, L - k * PAGE)
                flag[pg, :rows] = 0
        if kv_dtype == "bf16":
            lib().fill_rows_u16(_ptr(kv), _ptr(flag), P * PAGE, D_QK, 0x7FC0)
        else:
            lib().fill_rows_u8(_ptr(kv), _ptr(flag), P * PAGE, D_QK, 0x7F)
            kv_scale[flag.astype(bool)] = np.nan
    w_uv = None
    if with_w_uv:
        w_uv = normal_bf16(seed, S_WUV, (num_heads, D_V, D_UV), w_sigma)
    return Workload(name=name, batch=batch, q_len=q_len, num_heads=num_heads,
                    seq_lens=seq_lens, num_shards=num_shards, layout=layout,
                    kv_dtype=kv_dtype, causal=causal, seed=seed, q=q, kv=kv,
                    kv_scale=kv_scale, block_table=bt, w_uv=w_uv,
                    q_lens=None if q_lens is None else np.asarray(q_lens, dtype=np.int32))


def local_shard_cache(w: Workload, num_shards: int, shard: int, layout: str, seed: int = 0):
    """The slice of workload ``w``'s cache that shard ``shard`` of
    ``num_shards`` holds on its own GPU in a multi-GPU deployment: only the
    shard's token positions, in order, packed 64 to a page into a fresh page
    pool (scattered by a seeded permutation).  Interleaved shards own
    positions t = shard, shard + N, ...; contiguous shards own
    [shard * c, min((shard + 1) * c, L)), c = ceil(L / N).  Rows of the pool
    that hold no token are NaN-poisoned.

    Returns dict(kv, kv_scale, block_table, local_lens): the local cache in
    the same dtypes as ``w``, the local block table [B, max local pages] and
    each request's local token count.  The global lengths stay ``w.seq_lens``.
    """
    N, s = int(num_shards), int(shard)
    toks = []
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        if layout == "interleaved":
            t = np.arange(s, L, N, dtype=np.int64)
        elif layout == "contiguous":
            c = -(-L // N)
            t = np.arange(s * c, min((s + 1) * c, L), dtype=np.int64)
        else:
            raise ValueError(layout)
        toks.append(t)
    npages = [-(-len(t) // PAGE) for t in toks]
    P = max(1, sum(npages))
    perm = permutation(seed + 7919 * (s + 1), S_PERM + 50, P)
    kv = np.empty((P, PAGE, D_QK), dtype=w.kv.dtype)
    kv[...] = 0x7FC0 if w.kv.dtype == np.uint16 else 0x7F
    kv_scale = None
    if w.kv_scale is not None:
        kv_scale = np.full((P, PAGE), np.nan, dtype=np.float32)
    bt = np.full((w.batch, max(1, max(npages))), -1, dtype=np.int32)
    off = 0
    for b, t in enumerate(toks):
        n = npages[b]
        pages = perm[off:off + n]
        off += n
        bt[b, :n] = pages
        if len(t) == 0:
            continue
        k = np.arange(len(t))
        src_page = w.block_table[b, t // PAGE]
        src_row = t % PAGE
        kv[pages[k // PAGE], k % PAGE] = w.kv[src_page, src_row]
        if kv_scale is not None:
            kv_scale[pages[k // PAGE], k % PAGE] = w.kv_scale[src_page, src_row]
    local_lens = np.array([len(t) for t in toks], dtype=np.int32)
    return dict(kv=kv, kv_scale=kv_scale, block_table=bt, local_lens=local_lens)


@dataclass
class GqaWorkload:
    """A grouped-query-attention decode batch: Hkv KV heads of width D shared
    by groups of H / Hkv consecutive query heads, separate K and V caches."""
    name: str
    batch: int
    q_len: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    seq_lens: np.ndarray               # int32 [B]
    num_shards: int
    layout: str
    causal: bool
    seed: int
    q: np.ndarray = None               # uint16 (bf16 bits) [B, q_len, H, D]
    k_cache: np.ndarray = None         # uint16 [P, 64, Hkv, D]
    v_cache: np.ndarray = None         # uint16 [P, 64, Hkv, D]
    block_table: np.ndarray = None     # int32 [B, max_pages]
    softmax_scale: float = 0.0

    @property
    def num_pages(self):
        return self.k_cache.shape[0]

    @property
    def total_tokens(self):
        return int(np.sum(self.seq_lens.astype(np.int64)))

    def kv_bytes(self):
        """K and V bytes one full pass reads: every token < L_b once, all KV
        heads (2 * Hkv * D bf16 values per token)."""
        return self.total_tokens * 2 * self.num_kv_heads * self.head_dim * 2


def build_gqa_workload(name, batch, q_len, num_heads, num_kv_heads, head_dim, seq_lens,
                       num_shards, layout, causal, seed, q_sigma=0.5, kv_sigma=0.5,
                       extra_pages=0, poison=False, pinned=False):
    """Generate a GQA batch.  Pages are scattered by a seeded permutation of
    the pool as for the latent cache; ``poison`` fills rows past each
    request's end and unreferenced pages with NaN."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (batch,) and num_heads % num_kv_heads == 0
    pages_per = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    P = int(pages_per.sum()) + extra_pages
    perm = permutation(seed, S_PERM, max(P, 1))
    bt = np.full((batch, max(1, int(pages_per.max()))), -1, dtype=np.int32)
    off = 0
    for b in range(batch):
        n = int(pages_per[b])
        bt[b, :n] = perm[off:off + n]
        off += n

    def alloc(shape):
        if pinned:
            import torch
            return torch.empty(shape, dtype=torch.int16, pin_memory=True).numpy().view(np.uint16)
        return np.empty(shape, dtype=np.uint16)

    D, Hkv = head_dim, num_kv_heads
    q = alloc((batch, q_len, num_heads, D))
    normal_bf16(seed, S_Q, q.shape, q_sigma, out=q)
    k = alloc((max(P, 1), PAGE, Hkv, D))
    normal_bf16(seed, S_KV, k.shape, kv_sigma, out=k)
    v = alloc((max(P, 1), PAGE, Hkv, D))
    normal_bf16(seed, S_KV + 10, v.shape, kv_sigma, out=v)
    if poison:
        used = np.zeros((max(P, 1), PAGE), dtype=bool)
        for b in range(batch):
            L = int(seq_lens[b])
            for kk in range(int(pages_per[b])):
                used[bt[b, kk], :min(PAGE, L - kk * PAGE)] = True
        k[~used] = 0x7FC0
        v[~used] = 0x7FC0
    return GqaWorkload(name=name, batch=batch, q_len=q_len, num_heads=num_heads,
                       num_kv_heads=Hkv, head_dim=D, seq_lens=seq_lens,
                       num_shards=num_shards, layout=layout, causal=causal, seed=seed, q=q,
                       k_cache=k, v_cache=v, block_table=bt,
                       softmax_scale=1.0 / math.sqrt(D))


GQA_CONFIG_NAME = "gqa-agentic-b32-h64-kv4-d128-n2"


def config_gqa_workload(pinned=False):
    """Grouped-query decode over the bimodal agentic length mix: 32 requests,
    64 query heads sharing 4 KV heads of width 128 (groups of 16), bf16 K/V,
    2 interleaved shards (the GQA backend's DCP degree is bounded by the
    KV-head duplication factor)."""
    return build_gqa_workload(GQA_CONFIG_NAME, 32, 1, 64, 4, 128, agentic_lengths(6, 32), 2,
                              "interleaved", False, seed=6, pinned=pinned)


CONFIG_NAMES = {
    1: "tiny-b1-h16-l1024-n2-interleaved",
    2: "bimodal-agentic-b32-h64-n4-interleaved",
    3: "shard-sweep-b64-h64-l16k-96k",
    4: "spec-verify-b16-h64-q9-l8000-causal-n2",
    5: "longtail-fp8-b4-h64-l1m-n8-fused-wuv",
}


def config_params(cfg: int):
    """Arguments of build_workload for the five benchmark configurations."""
    if cfg == 1:
        return dict(name=CONFIG_NAMES[1], batch=1, q_len=1, num_heads=16, seq_lens=[1024],
                    num_shards=2, layout="interleaved", kv_dtype="bf16", causal=False, seed=1,
                    q_sigma=0.5, kv_sigma=0.5)
    if cfg == 2:
        return dict(name=CONFIG_NAMES[2], batch=32, q_len=1, num_heads=64,
                    seq_lens=agentic_lengths(2, 32), num_shards=4, layout="interleaved",
                    kv_dtype="bf16", causal=False, seed=2)
    if cfg == 3:
        return dict(name=CONFIG_NAMES[3], batch=64, q_len=1, num_heads=64,
                    seq_lens=uniform_lengths(3, 64, 16384, 98304), num_shards=1,
                    layout="interleaved", kv_dtype="bf16", causal=False, seed=3)
    if cfg == 4:
        return dict(name=CONFIG_NAMES[4], batch=16, q_len=9, num_heads=64, seq_lens=[8000] * 16,
                    num_shards=2, layout="interleaved", kv_dtype="bf16", causal=True, seed=4)
    if cfg == 5:
        return dict(name=CONFIG_NAMES[5], batch=4, q_len=1, num_heads=64,
                    seq_lens=[1048576, 262144, 131072, 65536], num_shards=8,
                    layout="interleaved", kv_dtype="fp8", causal=False, seed=5,
                    q_sigma=0.5, kv_sigma=1.0, with_w_uv=True, w_sigma=0.02)
    raise ValueError(cfg)


def config_workload(cfg: int, num_shards=None, layout=None, pinned=False, **kw):
    """The five benchmark configurations, generated from their seeds."""
    p = config_params(cfg)
    if num_shards:
        p["num_shards"] = num_shards
    if layout:
        p["layout"] = layout
    p.update(kw)
    return build_workload(pinned=pinned, **p)
