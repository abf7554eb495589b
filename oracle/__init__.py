"""fp64 CPU oracle for sequence-sharded MLA decode (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It shares no code with the CUDA path.
The arithmetic lives in ``mla_oracle.c``; this file marshals numpy arrays.
See the header of ``mla_oracle.c`` for the definition it follows and the
pins that check it.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

D_QK, D_V, D_UV = 576, 512, 128
LAYOUTS = {"interleaved": 0, "contiguous": 1}
_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build.build())
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_attend.argtypes = [vp, i32, i32, i32, vp, vp, i32, i32, vp, i32, vp, vp,
                                    i32, dbl, i32, i32, i32, vp, i64, vp, vp]
        L.oracle_attend.restype = i32
        L.oracle_gqa_attend.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, i32, vp,
                                        i32, dbl, i32, i32, i32, vp, i64, vp, vp]
        L.oracle_gqa_attend.restype = i32
        L.oracle_lse_merge.argtypes = [vp, vp, i32, i64, i32, vp, vp]
        L.oracle_lse_merge.restype = None
        L.oracle_project_wuv.argtypes = [vp, vp, vp, i64, vp]
        L.oracle_project_wuv.restype = None
        L.oracle_e4m3_decode.argtypes = [vp, ctypes.c_size_t, vp]
        L.oracle_e4m3_decode.restype = None
        L.oracle_bf16_decode.argtypes = [vp, ctypes.c_size_t, vp]
        L.oracle_bf16_decode.restype = None
        L.oracle_token_owner.argtypes = [ctypes.c_long, ctypes.c_long, i32, i32]
        L.oracle_token_owner.restype = i32
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = i32
        L.oracle_set_threads.argtypes = [i32]
        L.oracle_set_threads.restype = None
        _LIB = L
    return _LIB


def _p(a):
    if a is None:
        return None
    assert a.flags.c_contiguous, "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def attend(w, shard=-1, num_shards=None, layout=None, rows=None, q=None, seq_lens=None,
           block_table=None, kv=None, kv_scale=None, q_lens=None):
    """(out [n,512] fp64, lse [n] fp64) for query rows of workload ``w``.

    ``rows`` are flattened (b * q_len + i) * H + h indices (None = all rows).
    ``shard`` < 0 gives unsharded attention; otherwise shard ``shard`` of
    ``num_shards`` under ``layout``.  Individual tensors may be overridden.
    ``q_lens`` (default ``w.q_lens``): per-request query counts of a padded
    batch (rows i >= q_lens[b] are padding: lse -inf, out 0).
    """
    q = w.q if q is None else q
    seq_lens = w.seq_lens if seq_lens is None else seq_lens
    block_table = w.block_table if block_table is None else block_table
    kv = w.kv if kv is None else kv
    kv_scale = w.kv_scale if kv_scale is None else kv_scale
    if q_lens is None and w is not None:
        q_lens = getattr(w, "q_lens", None)
    if q_lens is not None:
        q_lens = np.ascontiguousarray(q_lens, dtype=np.int32)
    B, q_len, H = q.shape[0], q.shape[1], q.shape[2]
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    fp8 = 1 if kv.dtype == np.uint8 else 0
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.size
    else:
        n = B * q_len * H
    out = np.zeros((n, D_V), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    ns = num_shards if num_shards is not None else (w.num_shards if w is not None else 1)
    lay = LAYOUTS[layout if layout is not None else (w.layout if w is not None else "interleaved")]
    scale = w.softmax_scale if w is not None else 1.0 / np.sqrt(192.0)
    causal = int(w.causal) if w is not None else 0
    st = lib().oracle_attend(_p(q), B, q_len, H, _p(kv), _p(kv_scale), fp8, kv.shape[0],
                             _p(block_table), block_table.shape[1], _p(seq_lens), _p(q_lens),
                             causal,
                             float(scale), int(shard), int(ns), lay, _p(rows), n,
                             _p(out), _p(lse))
    if st != 0:
        raise RuntimeError(f"oracle_attend failed with status {st}")
    return out, lse


def gqa_attend(w, shard=-1, num_shards=None, layout=None, rows=None):
    """(out [n, D] fp64, lse [n] fp64) for query rows of GQA workload ``w``
    (rows = (b * q_len + i) * H + h; None = all)."""
    B, q_len, H, D = w.q.shape
    seq_lens = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(w.block_table, dtype=np.int32)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.size
    else:
        n = B * q_len * H
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    ns = num_shards if num_shards is not None else w.num_shards
    lay = LAYOUTS[layout if layout is not None else w.layout]
    st = lib().oracle_gqa_attend(_p(w.q), B, q_len, H, w.num_kv_heads, D, _p(w.k_cache),
                                 _p(w.v_cache), w.k_cache.shape[0], _p(bt), bt.shape[1],
                                 _p(seq_lens), int(w.causal), float(w.softmax_scale), int(shard),
                                 int(ns), lay, _p(rows), n, _p(out), _p(lse))
    if st != 0:
        raise RuntimeError(f"oracle_gqa_attend failed with status {st}")
    return out, lse


def lse_merge(outs, lses):
    """Merge shard partials: outs [N, rows, dim], lses [N, rows] (fp64)."""
    outs = np.ascontiguousarray(outs, dtype=np.float64)
    lses = np.ascontiguousarray(lses, dtype=np.float64)
    N, rows = lses.shape
    dim = outs.shape[-1]
    out = np.zeros((rows, dim), dtype=np.float64)
    lse = np.zeros((rows,), dtype=np.float64)
    lib().oracle_lse_merge(_p(outs), _p(lses), N, rows, dim, _p(out), _p(lse))
    return out, lse


def project_wuv(out, heads, w_uv):
    out = np.ascontiguousarray(out, dtype=np.float64)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    w_uv = np.ascontiguousarray(w_uv, dtype=np.uint16)
    y = np.zeros((out.shape[0], D_UV), dtype=np.float64)
    lib().oracle_project_wuv(_p(out), _p(heads), _p(w_uv), out.shape[0], _p(y))
    return y


def e4m3_decode(codes):
    codes = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    out = np.empty(codes.shape, dtype=np.float64)
    lib().oracle_e4m3_decode(_p(codes), codes.size, _p(out))
    return out


def bf16_decode(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.empty(bits.shape, dtype=np.float64)
    lib().oracle_bf16_decode(_p(bits), bits.size, _p(out))
    return out


def token_owner(t, L, num_shards, layout):
    """Shard that owns token ``t`` of an ``L``-token context (-1 if none)."""
    return int(lib().oracle_token_owner(int(t), int(L), int(num_shards), LAYOUTS[layout]))


def num_threads():
    return int(lib().oracle_num_threads())


def set_threads(n=0):
    """Host threads of later oracle calls: n > 0 that many, 0 the default."""
    lib().oracle_set_threads(int(n))


def reference_step(w, rows=None):
    """The whole decode step as the oracle defines it: unsharded attention,
    then the optional per-head W_UV projection.  Returns (out, lse, y)."""
    out, lse = attend(w, shard=-1, rows=rows)
    y = None
    if w.w_uv is not None:
        if rows is None:
            heads = np.tile(np.arange(w.num_heads, dtype=np.int32), w.batch * w.q_len)
        else:
            heads = (np.asarray(rows) % w.num_heads).astype(np.int32)
        y = project_wuv(out, heads, w.w_uv)
    return out, lse, y
