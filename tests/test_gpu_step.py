"""GPU parity of the whole single-GPU decode step (mla_decode_step): every
shard's partial attention and the LSE combine in one call, split pieces
merged inside the combine.  Compared element by element with the fp64
oracle's unsharded attention (and W_UV projection); the shard invariant of
"Decode Context Parallelism" section 4.1 says the two must agree."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from _helpers import REL_OUT, TOL_LSE, TOL_OUT, bf16_to_np, check_close, to_device

pytestmark = pytest.mark.gpu


def run_step(w, dev, layout=None, with_wuv=False):
    import torch
    import sequence_sharded_mla_gb300 as mla
    t = to_device(w, dev)
    out, lse, ws = mla.mla_decode_step(t["q"], t["kv"], t["block_table"], t["seq_lens"],
                                       w.num_shards, layout or w.layout, kv_scale=t["kv_scale"],
                                       causal=w.causal, softmax_scale=w.softmax_scale,
                                       w_uv=t["w_uv"] if with_wuv else None, q_lens=t["q_lens"])
    torch.cuda.synchronize()
    assert mla.mla_get_device_error(ws) == 0
    return out, lse


def check_step(w, dev, with_wuv=False):
    rows = w.batch * w.q_len * w.num_heads
    out, lse = run_step(w, dev, with_wuv=with_wuv)
    ref, ref_lse, ref_y = oracle.reference_step(w)
    check_close(lse.cpu().numpy().reshape(rows), ref_lse, TOL_LSE, "lse")
    if with_wuv:
        check_close(bf16_to_np(out).reshape(rows, 128), ref_y, TOL_OUT, "y", rel=REL_OUT)
    else:
        check_close(bf16_to_np(out).reshape(rows, 512), ref, TOL_OUT, "out", rel=REL_OUT)


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_step_ragged_split_units(dev, layout, N):
    """Long contexts next to short ones: the stream-K split cuts the long
    units into pieces that the combine merges with the other shards."""
    lens = [1, 63, 64, 65, 3000, 40000, 777]
    w = mi.build_workload("step", len(lens), 1, 64, lens, N, layout, "bf16", False,
                          seed=1000 + N, poison=True, extra_pages=3)
    check_step(w, dev)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_step_fused_wuv(dev, kv_dtype):
    lens = [70000, 5, 9000, 130, 33000]
    w = mi.build_workload("step-wuv", len(lens), 1, 64, lens, 8, "interleaved", kv_dtype, False,
                          seed=1010, with_w_uv=True, poison=True,
                          kv_sigma=1.0 if kv_dtype == "fp8" else 0.5)
    check_step(w, dev, with_wuv=True)


def test_step_wuv_many_rows_per_head(dev):
    """More query rows per head than one cluster's row block (8), causal."""
    lens = [300, 2000, 70, 1500]
    w = mi.build_workload("step-wuv9", len(lens), 9, 16, lens, 2, "interleaved", "bf16", True,
                          seed=1011, with_w_uv=True)
    check_step(w, dev, with_wuv=True)


@pytest.mark.parametrize("kv_dtype,B,q_len,q_lens", [
    ("bf16", 8, 9, None),                                   # 72 rows per head: one ragged block
    ("fp8", 16, 9, None),                                   # 144: a full block and a ragged one
    ("bf16", 16, 5, [5, 1, 3, 5, 2, 5, 4, 1, 5, 5, 3, 2, 1, 5, 4, 5]),   # padding rows
])
def test_step_wuv_tensor_core_projection(dev, kv_dtype, B, q_len, q_lens):
    """64 or more query rows per head: the combine writes o in bf16 and the
    W_UV projection runs as one tcgen05 GEMM per head in blocks of 128 rows."""
    lens = [37 + 911 * b % 3000 for b in range(B)]
    w = mi.build_workload("step-wuv-tc", B, q_len, 32, lens, 2, "interleaved", kv_dtype, True,
                          seed=1020 + B + q_len, with_w_uv=True, poison=True, q_lens=q_lens,
                          kv_sigma=1.0 if kv_dtype == "fp8" else 0.5)
    assert B * q_len >= 64
    check_step(w, dev, with_wuv=True)


def test_step_causal_and_padded_query_counts(dev):
    lens = [8000, 20, 3, 4100]
    w = mi.build_workload("step-q", len(lens), 9, 64, lens, 2, "interleaved", "bf16", True,
                          seed=1020, q_lens=[9, 3, 1, 5])
    check_step(w, dev)


def test_step_empty_shards_and_tiny_contexts(dev):
    w = mi.build_workload("step-empty", 3, 1, 16, [1, 3, 7], 8, "contiguous", "bf16", False,
                          seed=1030)
    check_step(w, dev)


def test_step_matches_partial_then_combine(dev):
    """The step equals mla_decode_partial + mla_shard_combine up to the
    rounding order of the merge (same pieces, merged at once)."""
    import sequence_sharded_mla_gb300 as mla
    from _helpers import run_gpu
    lens = [50000, 100, 20000, 4]
    w = mi.build_workload("step-eq", len(lens), 1, 64, lens, 4, "interleaved", "bf16", False,
                          seed=1040)
    a = run_gpu(w, dev)
    out, lse = run_step(w, dev)
    rows = w.batch * w.num_heads
    check_close(bf16_to_np(out).reshape(rows, 512), bf16_to_np(a["out"]).reshape(rows, 512),
                TOL_OUT, "out vs two-call", rel=REL_OUT)
    check_close(lse.cpu().numpy().reshape(rows), a["lse"].cpu().numpy().reshape(rows), 1e-5,
                "lse vs two-call")


def test_step_is_deterministic(dev):
    import torch
    lens = [60000, 10, 9000]
    w = mi.build_workload("step-det", len(lens), 1, 64, lens, 4, "interleaved", "bf16", False,
                          seed=1050)
    a, la = run_step(w, dev)
    b, lb = run_step(w, dev)
    assert torch.equal(a, b) and torch.equal(la, lb)
