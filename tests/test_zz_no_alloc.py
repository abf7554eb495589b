"""mla_decode_partial_noalloc: the partial-attention call for callers that
cannot allocate device memory (for instance while a serving engine's pool
owns the whole GPU, or inside allocator callbacks).  It runs on the
library's fixed scratch buffer instead of a caller workspace.

The results must match the ordinary workspace-taking entry point within the
parity tolerance, on two calls in a row (the scratch keeps the previous
call's contents), and shapes that do not fit the scratch must be refused
before anything is launched.  Collected last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from _helpers import REL_OUT, TOL_LSE, TOL_OUT, check_close, to_device

pytestmark = pytest.mark.gpu


def _noalloc_call(mla, t, w, N, layout, out, lse):
    """Call the C entry point directly through ctypes."""
    import torch
    L = mla.lib()
    sh = mla.mla_shape(w.batch, w.q_len, w.num_heads, int(w.causal), float(w.softmax_scale))
    pages = mla.mla_kv_pages(t["kv"].data_ptr(), None, mla.KV_BF16, t["kv"].shape[0],
                             t["kv"].shape[1])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.mla_decode_partial_noalloc(
        ctypes.c_void_p(t["q"].data_ptr()), ctypes.byref(pages),
        ctypes.c_void_p(t["block_table"].data_ptr()), t["block_table"].shape[1],
        ctypes.c_void_p(t["seq_lens"].data_ptr()), ctypes.byref(sh), -1, N,
        mla.LAYOUTS[layout], ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        stream)


@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
def test_noalloc_matches_workspace_entry_point_twice(layout):
    import torch
    import sequence_sharded_mla_gb300 as mla
    dev = torch.device("cuda:0")
    # ragged contexts and enough tiles that work units are split across CTAs,
    # so the split-piece part of the scratch is exercised
    w = mi.build_workload("noalloc", 4, 1, 64, [5000, 70, 20000, 1], 4, layout, "bf16", False,
                          seed=900, poison=True, extra_pages=2)
    t = to_device(w, dev)
    ref, ref_lse, _ = mla.mla_decode_partial(t["q"], t["kv"], t["block_table"], t["seq_lens"],
                                             4, layout)
    torch.cuda.synchronize()
    rows = w.batch * w.q_len * w.num_heads
    ref_np = ref.cpu().numpy().reshape(4, rows, 512)
    ref_lse_np = ref_lse.cpu().numpy().reshape(4, rows)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _noalloc_call(mla, t, w, 4, layout, out, lse)
        assert st == 0, mla.mla_status_string(st)
        torch.cuda.synchronize()
        got = out.cpu().numpy().reshape(4, rows, 512)
        got_lse = lse.cpu().numpy().reshape(4, rows)
        for s in range(4):
            check_close(got[s], ref_np[s], TOL_OUT, f"call {call} shard {s}", rel=REL_OUT)
            check_close(got_lse[s], ref_lse_np[s], TOL_LSE, f"call {call} lse shard {s}")


@pytest.mark.gpu
def test_noalloc_second_call_after_other_entry_points():
    """The fixed scratch is independent of caller workspaces: interleaving a
    workspace call between two scratch calls changes nothing."""
    import torch
    import sequence_sharded_mla_gb300 as mla
    dev = torch.device("cuda:0")
    w = mi.build_workload("noalloc2", 2, 9, 16, [300, 1000], 2, "interleaved", "bf16", True,
                          seed=901)
    t = to_device(w, dev)
    out1 = torch.empty((2, 2, 9, 16, 512), dtype=torch.float32, device=dev)
    lse1 = torch.empty((2, 2, 9, 16), dtype=torch.float32, device=dev)
    assert _noalloc_call(mla, t, w, 2, "interleaved", out1, lse1) == 0
    ref, ref_lse, _ = mla.mla_decode_partial(t["q"], t["kv"], t["block_table"], t["seq_lens"], 2,
                                             "interleaved", causal=True)
    out2 = torch.empty_like(out1)
    lse2 = torch.empty_like(lse1)
    assert _noalloc_call(mla, t, w, 2, "interleaved", out2, lse2) == 0
    torch.cuda.synchronize()
    for o, l in ((out1, lse1), (out2, lse2)):
        check_close(o.cpu().numpy(), ref.cpu().numpy(), TOL_OUT, "out", rel=REL_OUT)
        check_close(l.cpu().numpy(), ref_lse.cpu().numpy(), TOL_LSE, "lse")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_noalloc_matches_the_oracle(kv_dtype):
    """Every shard's partial from the scratch-backed call against the fp64
    oracle, bf16 and fp8 caches, with split work units (long contexts)."""
    import torch
    import sequence_sharded_mla_gb300 as mla
    dev = torch.device("cuda:0")
    w = mi.build_workload("noalloc-oracle", 3, 1, 32, [4100, 70, 9000], 4, "interleaved",
                          kv_dtype, False, seed=902, poison=True, extra_pages=2,
                          kv_sigma=1.0 if kv_dtype == "fp8" else 0.5)
    t = to_device(w, dev)
    rows = w.batch * w.q_len * w.num_heads
    for call in range(2):
        out, lse = mla.mla_decode_partial_noalloc(t["q"], t["kv"], t["block_table"],
                                                  t["seq_lens"], 4, "interleaved",
                                                  kv_scale=t["kv_scale"])
        assert mla.mla_get_device_error_noalloc() == 0
        got = out.cpu().numpy().reshape(4, rows, 512)
        got_lse = lse.cpu().numpy().reshape(4, rows)
        for s in range(4):
            ro, rl = oracle.attend(w, shard=s, num_shards=4, layout="interleaved")
            check_close(got[s], ro, TOL_OUT, f"call {call} shard {s}", rel=REL_OUT)
            check_close(got_lse[s], rl, TOL_LSE, f"call {call} lse shard {s}")


def test_noalloc_local_shard_cache_matches_the_oracle():
    """The per-GPU call of a multi-GPU deployment (one shard, a cache that
    holds only that shard's positions, causal verify rows) on the scratch."""
    import torch
    import sequence_sharded_mla_gb300 as mla
    dev = torch.device("cuda:0")
    lens = [1, 300, 5000]
    w = mi.build_workload("noalloc-local", len(lens), 2, 32, lens, 3, "interleaved", "bf16",
                          True, seed=903, poison=True)
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    rows = w.batch * w.q_len * w.num_heads
    for s in range(3):
        d = mi.local_shard_cache(w, 3, s, "interleaved", seed=s)
        kv = torch.from_numpy(d["kv"].view(np.int16)).view(torch.bfloat16).to(dev)
        bt = torch.from_numpy(d["block_table"]).to(dev)
        out, lse = mla.mla_decode_partial_noalloc(q, kv, bt, sl, 3, "interleaved_local",
                                                  shard_id=s, causal=True)
        assert mla.mla_get_device_error_noalloc() == 0
        ro, rl = oracle.attend(w, shard=s, num_shards=3, layout="interleaved")
        check_close(out.cpu().numpy().reshape(rows, 512), ro, TOL_OUT, f"local shard {s}",
                    rel=REL_OUT)
        check_close(lse.cpu().numpy().reshape(rows), rl, TOL_LSE, f"local lse {s}")


def test_noalloc_reports_a_bad_block_table_page():
    """A block-table entry outside the page pool is read as zeros and
    reported through the scratch's error word; reading clears it."""
    import torch
    import sequence_sharded_mla_gb300 as mla
    dev = torch.device("cuda:0")
    w = mi.build_workload("noalloc-bad", 2, 1, 16, [200, 64], 2, "interleaved", "bf16", False,
                          seed=904)
    w.block_table[0, 2] = w.num_pages + 100
    t = to_device(w, dev)
    out, lse = mla.mla_decode_partial_noalloc(t["q"], t["kv"], t["block_table"], t["seq_lens"],
                                              2, "interleaved")
    assert mla.mla_get_device_error_noalloc() == -5          # MLA_ERR_DEVICE_BOUNDS
    assert mla.mla_get_device_error_noalloc() == 0
    assert np.all(np.isfinite(out.cpu().numpy()))
