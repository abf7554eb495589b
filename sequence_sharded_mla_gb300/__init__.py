"""Sequence-sharded MLA decode for GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/mla_dcp.h``: it checks tensor
dtypes/devices, allocates outputs and workspace with PyTorch and passes raw
pointers and the current CUDA stream to ``libmla_dcp.so``.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.
If the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import build as _build

D_QK, D_V, D_UV, PAGE = 576, 512, 128, 64
ALL_SHARDS = -1
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)
LAYOUTS = {"interleaved": 0, "contiguous": 1, "interleaved_local": 2, "contiguous_local": 3}
KV_BF16, KV_FP8 = 0, 1

STATUS = {0: "MLA_OK", -1: "MLA_ERR_INVALID", -2: "MLA_ERR_UNSUPPORTED", -3: "MLA_ERR_CUDA",
          -4: "MLA_ERR_TIMEOUT", -5: "MLA_ERR_DEVICE_BOUNDS", -6: "MLA_ERR_WORKSPACE",
          -7: "MLA_ERR_RANGE"}


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class mla_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("q_len", ctypes.c_int), ("num_heads", ctypes.c_int),
                ("causal", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("q_lens", ctypes.c_void_p)]


class mla_kv_pages(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("page_size", ctypes.c_int)]


class gqa_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("q_len", ctypes.c_int), ("num_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("causal", ctypes.c_int), ("softmax_scale", ctypes.c_float)]


class gqa_kv_pages(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_pages", ctypes.c_int),
                ("page_size", ctypes.c_int)]


_LIB = None
EXPORTS = ("mla_decode_partial", "mla_decode_partial_noalloc", "mla_decode_partial_dcp",
           "mla_shard_combine",
           "mla_decode_step", "mla_decode_step_workspace_size",
           "mla_workspace_size", "mla_get_device_error", "mla_get_device_error_noalloc",
           "mla_set_wait_budget_ns", "mla_set_withhold_query", "mla_set_profile_events",
           "mla_status_string",
           "mla_version", "gqa_workspace_size", "gqa_decode_partial", "gqa_shard_combine")


def lib():
    """Load (building first if the sources are newer) ``libmla_dcp.so``."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.mla_decode_partial.argtypes = [vp, ctypes.POINTER(mla_kv_pages), vp, i32, vp,
                                         ctypes.POINTER(mla_shape), i32, i32, i32, vp, vp, vp,
                                         sz, vp]
        L.mla_decode_partial.restype = i32
        L.mla_decode_partial_dcp.argtypes = [vp, i32, i32, ctypes.POINTER(mla_kv_pages), vp, i32,
                                             vp, ctypes.POINTER(mla_shape), i32, i32, i32, vp, vp,
                                             vp, sz, vp]
        L.mla_decode_partial_dcp.restype = i32
        L.mla_decode_partial_noalloc.argtypes = [vp, ctypes.POINTER(mla_kv_pages), vp, i32, vp,
                                                 ctypes.POINTER(mla_shape), i32, i32, i32, vp,
                                                 vp, vp]
        L.mla_decode_partial_noalloc.restype = i32
        L.mla_shard_combine.argtypes = [vp, vp, i32, ctypes.POINTER(mla_shape), vp, vp, vp, vp]
        L.mla_shard_combine.restype = i32
        L.mla_decode_step.argtypes = [vp, ctypes.POINTER(mla_kv_pages), vp, i32, vp,
                                      ctypes.POINTER(mla_shape), i32, i32, vp, vp, vp, vp, sz,
                                      vp]
        L.mla_decode_step.restype = i32
        L.mla_decode_step_workspace_size.argtypes = [ctypes.POINTER(mla_shape), i32]
        L.mla_decode_step_workspace_size.restype = sz
        L.mla_workspace_size.argtypes = [ctypes.POINTER(mla_shape), i32, i32]
        L.mla_workspace_size.restype = sz
        L.mla_get_device_error.argtypes = [vp, vp]
        L.mla_get_device_error.restype = i32
        L.mla_get_device_error_noalloc.argtypes = [vp]
        L.mla_get_device_error_noalloc.restype = i32
        L.mla_set_wait_budget_ns.argtypes = [ctypes.c_ulonglong]
        L.mla_set_wait_budget_ns.restype = i32
        L.mla_set_withhold_query.argtypes = [i32]
        L.mla_set_withhold_query.restype = i32
        L.mla_set_profile_events.argtypes = [vp, vp]
        L.mla_set_profile_events.restype = i32
        L.mla_status_string.argtypes = [i32]
        L.mla_status_string.restype = ctypes.c_char_p
        L.mla_version.argtypes = []
        L.mla_version.restype = i32
        L.gqa_workspace_size.argtypes = [ctypes.POINTER(gqa_shape), i32, i32]
        L.gqa_workspace_size.restype = sz
        L.gqa_decode_partial.argtypes = [vp, ctypes.POINTER(gqa_kv_pages), vp, i32, vp,
                                         ctypes.POINTER(gqa_shape), i32, i32, i32, vp, vp, vp,
                                         sz, vp]
        L.gqa_decode_partial.restype = i32
        L.gqa_shard_combine.argtypes = [vp, vp, i32, ctypes.POINTER(gqa_shape), vp, vp, vp]
        L.gqa_shard_combine.restype = i32
        _LIB = L
    return _LIB


def _shape(batch, q_len, num_heads, causal, softmax_scale, q_lens=None):
    return mla_shape(int(batch), int(q_len), int(num_heads), int(bool(causal)),
                     float(softmax_scale), None if q_lens is None else q_lens.data_ptr())


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtypes, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def mla_workspace_size(batch, q_len, num_heads, num_shards, shard_id=ALL_SHARDS, causal=False,
                       softmax_scale=DEFAULT_SCALE) -> int:
    sh = _shape(batch, q_len, num_heads, causal, softmax_scale)
    return int(lib().mla_workspace_size(ctypes.byref(sh), int(num_shards), int(shard_id)))


def _kv_pages(kv, kv_scale, dev):
    """The mla_kv_pages descriptor of a bf16 or e4m3 cache (checked)."""
    if kv.dtype == torch.bfloat16:
        kv_dtype = KV_BF16
        if kv_scale is not None:
            raise ValueError("kv_scale is only for fp8 caches")
    elif kv.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        kv_dtype = KV_FP8
        if kv_scale is None:
            raise ValueError("fp8 caches need kv_scale")
        _check(kv_scale, "kv_scale", (torch.float32,), 2, dev)
    else:
        raise TypeError(f"kv dtype {kv.dtype} unsupported")
    _check(kv, "kv", (kv.dtype,), 3, dev)
    return mla_kv_pages(kv.data_ptr(), None if kv_scale is None else kv_scale.data_ptr(),
                        kv_dtype, kv.shape[0], kv.shape[1])


def mla_decode_partial(q, kv, block_table, seq_lens, num_shards, layout="interleaved",
                       shard_id=ALL_SHARDS, kv_scale=None, causal=False,
                       softmax_scale=DEFAULT_SCALE, out_partial=None, lse_partial=None,
                       workspace=None, stream=None, q_lens=None):
    """Per-shard partial attention; returns (out_partial, lse_partial, workspace).

    q: bf16 [B, q_len, H, 576]; kv: bf16 [P, 64, 576] or e4m3 codes
    (uint8 / float8_e4m3fn) [P, 64, 576] with kv_scale fp32 [P, 64];
    block_table: int32 [B, max_pages]; seq_lens: int32 [B] (device).
    out_partial: fp32 [n_out, B, q_len, H, 512]; lse_partial: fp32 [n_out, B, q_len, H].
    q_lens: optional int32 [B] (device) query tokens per request of a padded
    batch (rows i >= q_lens[b] are padding).
    """
    _check(q, "q", (torch.bfloat16,), 4)
    dev = q.device
    B, q_len, H, d = q.shape
    if d != D_QK:
        raise ValueError("q must be [B, q_len, H, 576]")
    pages = _kv_pages(kv, kv_scale, dev)
    _check(block_table, "block_table", (torch.int32,), 2, dev)
    _check(seq_lens, "seq_lens", (torch.int32,), 1, dev)
    n_out = num_shards if shard_id == ALL_SHARDS else 1
    if out_partial is None:
        out_partial = torch.empty((n_out, B, q_len, H, D_V), dtype=torch.float32, device=dev)
    if lse_partial is None:
        lse_partial = torch.empty((n_out, B, q_len, H), dtype=torch.float32, device=dev)
    _check(out_partial, "out_partial", (torch.float32,), 5, dev)
    _check(lse_partial, "lse_partial", (torch.float32,), 4, dev)
    if q_lens is not None:
        _check(q_lens, "q_lens", (torch.int32,), 1, dev)
    sh = _shape(B, q_len, H, causal, softmax_scale, q_lens)
    need = int(lib().mla_workspace_size(ctypes.byref(sh), int(num_shards), int(shard_id)))
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    st = lib().mla_decode_partial(_ptr(q), ctypes.byref(pages), _ptr(block_table),
                                  block_table.shape[1], _ptr(seq_lens), ctypes.byref(sh),
                                  int(shard_id), int(num_shards), LAYOUTS[layout],
                                  _ptr(out_partial), _ptr(lse_partial), _ptr(workspace),
                                  workspace.numel(), _stream_ptr(stream))
    if st != 0:
        raise MLAError(st, "mla_decode_partial")
    return out_partial, lse_partial, workspace


def mla_decode_partial_dcp(q_gathered, kv, block_table, seq_lens, rank,
                           layout="interleaved_local", batch_first=0, kv_scale=None,
                           causal=False, softmax_scale=DEFAULT_SCALE, out_send=None,
                           lse_send=None, workspace=None, stream=None, q_lens=None):
    """The per-rank call of a DCP step in the exchanges' own layouts; returns
    (out_send, lse_send, workspace).

    q_gathered: bf16 [N, B_total, q_len, H/N, 576], the all-gather of the N
    ranks' query heads; this call computes requests batch_first ..
    batch_first + len(seq_lens) - 1 of it over shard `rank` of N of this
    rank's cache (block_table, seq_lens, q_lens: those requests' rows).
    out_send: fp32 [N, B, q_len, H/N, 512], lse_send: fp32 [N, B, q_len, H/N]:
    slice k is this shard's partial of rank k's heads -- the all-to-all's send
    buffers.
    """
    _check(q_gathered, "q_gathered", (torch.bfloat16,), 5)
    dev = q_gathered.device
    N, B_total, q_len, Hl, d = q_gathered.shape
    if d != D_QK:
        raise ValueError("q_gathered must be [N, B_total, q_len, H/N, 576]")
    pages = _kv_pages(kv, kv_scale, dev)
    _check(block_table, "block_table", (torch.int32,), 2, dev)
    _check(seq_lens, "seq_lens", (torch.int32,), 1, dev)
    B = seq_lens.shape[0]
    if block_table.shape[0] != B:
        raise ValueError("block_table and seq_lens disagree on the number of requests")
    if out_send is None:
        out_send = torch.empty((N, B, q_len, Hl, D_V), dtype=torch.float32, device=dev)
    if lse_send is None:
        lse_send = torch.empty((N, B, q_len, Hl), dtype=torch.float32, device=dev)
    _check(out_send, "out_send", (torch.float32,), 5, dev)
    _check(lse_send, "lse_send", (torch.float32,), 4, dev)
    if q_lens is not None:
        _check(q_lens, "q_lens", (torch.int32,), 1, dev)
    sh = _shape(B, q_len, N * Hl, causal, softmax_scale, q_lens)
    need = int(lib().mla_workspace_size(ctypes.byref(sh), int(N), int(rank)))
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    st = lib().mla_decode_partial_dcp(_ptr(q_gathered), int(B_total), int(batch_first),
                                      ctypes.byref(pages), _ptr(block_table),
                                      block_table.shape[1], _ptr(seq_lens), ctypes.byref(sh),
                                      int(rank), int(N), LAYOUTS[layout], _ptr(out_send),
                                      _ptr(lse_send), _ptr(workspace), workspace.numel(),
                                      _stream_ptr(stream))
    if st != 0:
        raise MLAError(st, "mla_decode_partial_dcp")
    return out_send, lse_send, workspace


def mla_decode_step_workspace_size(batch, q_len, num_heads, num_shards) -> int:
    sh = _shape(batch, q_len, num_heads, False, DEFAULT_SCALE)
    return int(lib().mla_decode_step_workspace_size(ctypes.byref(sh), int(num_shards)))


def mla_decode_step(q, kv, block_table, seq_lens, num_shards, layout="interleaved",
                    kv_scale=None, causal=False, softmax_scale=DEFAULT_SCALE, w_uv=None,
                    out=None, lse_out=None, workspace=None, stream=None, q_lens=None):
    """One whole decode step on one GPU: all shards' partials and their LSE
    combine (optionally fused with W_UV); returns (out, lse_out, workspace).

    Inputs as for mla_decode_partial; w_uv: bf16 [H, 512, 128] or None.
    out: bf16 [B, q_len, H, 512] (or [.., 128] with w_uv); lse_out: fp32 [B, q_len, H].
    """
    _check(q, "q", (torch.bfloat16,), 4)
    dev = q.device
    B, q_len, H, d = q.shape
    if d != D_QK:
        raise ValueError("q must be [B, q_len, H, 576]")
    if kv.dtype == torch.bfloat16:
        kv_dtype = KV_BF16
        if kv_scale is not None:
            raise ValueError("kv_scale is only for fp8 caches")
    elif kv.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        kv_dtype = KV_FP8
        if kv_scale is None:
            raise ValueError("fp8 caches need kv_scale")
        _check(kv_scale, "kv_scale", (torch.float32,), 2, dev)
    else:
        raise TypeError(f"kv dtype {kv.dtype} unsupported")
    _check(kv, "kv", (kv.dtype,), 3, dev)
    _check(block_table, "block_table", (torch.int32,), 2, dev)
    _check(seq_lens, "seq_lens", (torch.int32,), 1, dev)
    if w_uv is not None:
        _check(w_uv, "w_uv", (torch.bfloat16,), 3, dev)
    if q_lens is not None:
        _check(q_lens, "q_lens", (torch.int32,), 1, dev)
    width = D_UV if w_uv is not None else D_V
    if out is None:
        out = torch.empty((B, q_len, H, width), dtype=torch.bfloat16, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    _check(out, "out", (torch.bfloat16,), 4, dev)
    _check(lse_out, "lse_out", (torch.float32,), 3, dev)
    sh = _shape(B, q_len, H, causal, softmax_scale, q_lens)
    need = int(lib().mla_decode_step_workspace_size(ctypes.byref(sh), int(num_shards)))
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    pages = mla_kv_pages(kv.data_ptr(), None if kv_scale is None else kv_scale.data_ptr(),
                         kv_dtype, kv.shape[0], kv.shape[1])
    st = lib().mla_decode_step(_ptr(q), ctypes.byref(pages), _ptr(block_table),
                               block_table.shape[1], _ptr(seq_lens), ctypes.byref(sh),
                               int(num_shards), LAYOUTS[layout], _ptr(w_uv), _ptr(out),
                               _ptr(lse_out), _ptr(workspace), workspace.numel(),
                               _stream_ptr(stream))
    if st != 0:
        raise MLAError(st, "mla_decode_step")
    return out, lse_out, workspace


def mla_decode_partial_noalloc(q, kv, block_table, seq_lens, num_shards, layout="interleaved",
                               shard_id=ALL_SHARDS, kv_scale=None, causal=False,
                               softmax_scale=DEFAULT_SCALE, out_partial=None, lse_partial=None,
                               stream=None, q_lens=None):
    """mla_decode_partial on the library's fixed scratch buffer (no workspace).

    For callers that may not allocate device memory; the output tensors are
    still supplied by (or allocated here for) the caller.  All calls on a
    device share one scratch buffer: keep calls on one stream.
    Returns (out_partial, lse_partial).
    """
    _check(q, "q", (torch.bfloat16,), 4)
    dev = q.device
    B, q_len, H, _ = q.shape
    if kv.dtype == torch.bfloat16:
        kv_dtype = KV_BF16
    elif kv.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        kv_dtype = KV_FP8
        _check(kv_scale, "kv_scale", (torch.float32,), 2, dev)
    else:
        raise TypeError(f"kv dtype {kv.dtype} unsupported")
    _check(kv, "kv", (kv.dtype,), 3, dev)
    _check(block_table, "block_table", (torch.int32,), 2, dev)
    _check(seq_lens, "seq_lens", (torch.int32,), 1, dev)
    n_out = num_shards if shard_id == ALL_SHARDS else 1
    if out_partial is None:
        out_partial = torch.empty((n_out, B, q_len, H, D_V), dtype=torch.float32, device=dev)
    if lse_partial is None:
        lse_partial = torch.empty((n_out, B, q_len, H), dtype=torch.float32, device=dev)
    _check(out_partial, "out_partial", (torch.float32,), 5, dev)
    _check(lse_partial, "lse_partial", (torch.float32,), 4, dev)
    if q_lens is not None:
        _check(q_lens, "q_lens", (torch.int32,), 1, dev)
    sh = _shape(B, q_len, H, causal, softmax_scale, q_lens)
    pages = mla_kv_pages(kv.data_ptr(), None if kv_scale is None else kv_scale.data_ptr(),
                         kv_dtype, kv.shape[0], kv.shape[1])
    st = lib().mla_decode_partial_noalloc(_ptr(q), ctypes.byref(pages), _ptr(block_table),
                                          block_table.shape[1], _ptr(seq_lens), ctypes.byref(sh),
                                          int(shard_id), int(num_shards), LAYOUTS[layout],
                                          _ptr(out_partial), _ptr(lse_partial),
                                          _stream_ptr(stream))
    if st != 0:
        raise MLAError(st, "mla_decode_partial_noalloc")
    return out_partial, lse_partial


def mla_shard_combine(partials, lses, w_uv=None, out=None, lse_out=None, stream=None,
                      causal=False, softmax_scale=DEFAULT_SCALE):
    """LSE combine (optionally fused with W_UV); returns (out, lse_out).

    partials: fp32 [N, B, q_len, H, 512]; lses: fp32 [N, B, q_len, H];
    w_uv: bf16 [H, 512, 128] or None.  out: bf16 [B, q_len, H, 512|128].
    """
    _check(partials, "partials", (torch.float32,), 5)
    dev = partials.device
    N, B, q_len, H, d = partials.shape
    _check(lses, "lses", (torch.float32,), 4, dev)
    if w_uv is not None:
        _check(w_uv, "w_uv", (torch.bfloat16,), 3, dev)
    width = D_UV if w_uv is not None else D_V
    if out is None:
        out = torch.empty((B, q_len, H, width), dtype=torch.bfloat16, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    sh = _shape(B, q_len, H, causal, softmax_scale)
    st = lib().mla_shard_combine(_ptr(partials), _ptr(lses), int(N), ctypes.byref(sh),
                                 _ptr(w_uv), _ptr(out), _ptr(lse_out), _stream_ptr(stream))
    if st != 0:
        raise MLAError(st, "mla_shard_combine")
    return out, lse_out


def mla_get_device_error(workspace, stream=None) -> int:
    """Sync the stream, read and clear the device error word; returns a status code."""
    return int(lib().mla_get_device_error(_ptr(workspace), _stream_ptr(stream)))


def mla_get_device_error_noalloc(stream=None) -> int:
    """Sync the stream, read and clear the error word of the fixed scratch
    used by mla_decode_partial_noalloc; returns a status code."""
    return int(lib().mla_get_device_error_noalloc(_stream_ptr(stream)))


def mla_set_wait_budget_ns(ns: int) -> None:
    """Testing aid: time limit (ns) of every device-side wait of later
    partial-attention launches; 0 restores the default (2 s)."""
    lib().mla_set_wait_budget_ns(int(ns))


def mla_set_withhold_query(on: bool) -> None:
    """Testing aid: while on, later partial-attention launches never load the
    first piece's query rows, so their waits run out (MLA_ERR_TIMEOUT)."""
    lib().mla_set_withhold_query(int(bool(on)))


def mla_set_profile_events(before=None, after=None) -> None:
    """Record two torch.cuda.Events around the partial-attention kernel of
    every later mla_decode_partial call (None, None stops).  The events are
    recorded once here on the current stream so that their CUDA handles exist."""
    if (before is None) != (after is None):
        raise ValueError("give both events or neither")
    if before is None:
        st = lib().mla_set_profile_events(None, None)
    else:
        for ev in (before, after):
            if ev.cuda_event == 0:
                ev.record()
        st = lib().mla_set_profile_events(ctypes.c_void_p(before.cuda_event),
                                          ctypes.c_void_p(after.cuda_event))
    if st != 0:
        raise MLAError(st, "mla_set_profile_events")


def mla_status_string(status: int) -> str:
    return lib().mla_status_string(int(status)).decode()


def mla_version() -> int:
    return int(lib().mla_version())


# --------------------------------------------------------------------- GQA
def _gqa_shape(batch, q_len, num_heads, num_kv_heads, head_dim, causal, softmax_scale):
    return gqa_shape(int(batch), int(q_len), int(num_heads), int(num_kv_heads), int(head_dim),
                     int(bool(causal)), float(softmax_scale))


def gqa_workspace_size(batch, q_len, num_heads, num_kv_heads, num_shards,
                       shard_id=ALL_SHARDS, head_dim=128, causal=False) -> int:
    sh = _gqa_shape(batch, q_len, num_heads, num_kv_heads, head_dim, causal, 1.0)
    return int(lib().gqa_workspace_size(ctypes.byref(sh), int(num_shards), int(shard_id)))


def gqa_decode_partial(q, k_cache, v_cache, block_table, seq_lens, num_shards,
                       layout="interleaved", shard_id=ALL_SHARDS, causal=False,
                       softmax_scale=None, out_partial=None, lse_partial=None, workspace=None,
                       stream=None):
    """Per-shard partial grouped-query attention; returns (out_partial, lse_partial, workspace).

    q: bf16 [B, q_len, H, D]; k_cache, v_cache: bf16 [P, 64, Hkv, D];
    block_table: int32 [B, max_pages]; seq_lens: int32 [B] (device).
    out_partial: fp32 [n_out, B, q_len, H, D]; lse_partial: fp32 [n_out, B, q_len, H].
    softmax_scale defaults to 1/sqrt(D).
    """
    _check(q, "q", (torch.bfloat16,), 4)
    dev = q.device
    B, q_len, H, D = q.shape
    _check(k_cache, "k_cache", (torch.bfloat16,), 4, dev)
    _check(v_cache, "v_cache", (torch.bfloat16,), 4, dev)
    if k_cache.shape != v_cache.shape or k_cache.shape[3] != D:
        raise ValueError("k_cache and v_cache must both be [P, 64, Hkv, D]")
    Hkv = k_cache.shape[2]
    _check(block_table, "block_table", (torch.int32,), 2, dev)
    _check(seq_lens, "seq_lens", (torch.int32,), 1, dev)
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else softmax_scale
    n_out = num_shards if shard_id == ALL_SHARDS else 1
    if out_partial is None:
        out_partial = torch.empty((n_out, B, q_len, H, D), dtype=torch.float32, device=dev)
    if lse_partial is None:
        lse_partial = torch.empty((n_out, B, q_len, H), dtype=torch.float32, device=dev)
    _check(out_partial, "out_partial", (torch.float32,), 5, dev)
    _check(lse_partial, "lse_partial", (torch.float32,), 4, dev)
    sh = _gqa_shape(B, q_len, H, Hkv, D, causal, scale)
    need = int(lib().gqa_workspace_size(ctypes.byref(sh), int(num_shards), int(shard_id)))
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=dev)
    pages = gqa_kv_pages(k_cache.data_ptr(), v_cache.data_ptr(), k_cache.shape[0],
                         k_cache.shape[1])
    st = lib().gqa_decode_partial(_ptr(q), ctypes.byref(pages), _ptr(block_table),
                                  block_table.shape[1], _ptr(seq_lens), ctypes.byref(sh),
                                  int(shard_id), int(num_shards), LAYOUTS[layout],
                                  _ptr(out_partial), _ptr(lse_partial), _ptr(workspace),
                                  workspace.numel(), _stream_ptr(stream))
    if st != 0:
        raise MLAError(st, "gqa_decode_partial")
    return out_partial, lse_partial, workspace


def gqa_shard_combine(partials, lses, out=None, lse_out=None, stream=None):
    """LSE combine of GQA shard partials fp32 [N, B, q_len, H, D] -> bf16
    [B, q_len, H, D] and fp32 lse [B, q_len, H]."""
    _check(partials, "partials", (torch.float32,), 5)
    dev = partials.device
    N, B, q_len, H, D = partials.shape
    _check(lses, "lses", (torch.float32,), 4, dev)
    if out is None:
        out = torch.empty((B, q_len, H, D), dtype=torch.bfloat16, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    sh = _gqa_shape(B, q_len, H, 1, D, False, 1.0)
    st = lib().gqa_shard_combine(_ptr(partials), _ptr(lses), int(N), ctypes.byref(sh), _ptr(out),
                                 _ptr(lse_out), _stream_ptr(stream))
    if st != 0:
        raise MLAError(st, "gqa_shard_combine")
    return out, lse_out
