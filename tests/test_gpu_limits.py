"""GPU parity at the edges of the supported sizes: one request of 4M tokens
(the largest context of the benchmark mixes) over 8 shards, a batch of 2048
short requests (8192 work units: several units per planning thread), and
128 heads x q_len 9 causal (18 row groups per request).  Sampled rows are
checked against the oracle; every other row against invariants that hold at
any size (finite, -inf pattern of empty rows)."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from _helpers import REL_OUT, TOL_LSE, TOL_OUT, bf16_to_np, check_close, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


def check_rows(w, res, rows, N, layout):
    R = w.batch * w.q_len * w.num_heads
    out = bf16_to_np(res["out"]).reshape(R, 512)
    lse = res["lse"].cpu().numpy().reshape(R)
    assert np.all(np.isfinite(out))
    ref, ref_lse = oracle.attend(w, shard=-1, rows=rows)
    check_close(out[rows], ref, TOL_OUT, "out", rel=REL_OUT)
    check_close(lse[rows], ref_lse, TOL_LSE, "lse")
    part = res["partial"].cpu().numpy().reshape(N, R, 512)
    lsep = res["lse_partial"].cpu().numpy().reshape(N, R)
    for s in range(N):
        po, pl = oracle.attend(w, shard=s, num_shards=N, layout=layout, rows=rows)
        check_close(part[s][rows], po, TOL_OUT, f"partial {s}", rel=REL_OUT)
        check_close(lsep[s][rows], pl, TOL_LSE, f"lse_partial {s}")


@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
def test_four_million_token_context(dev, layout):
    L = 4 * 1024 * 1024
    w = mi.build_workload("4m", 1, 1, 64, [L], 8, layout, "bf16", False, seed=900)
    res = run_gpu(w, dev)
    assert res["status"] == 0
    rows = np.array([0, 17, 40, 63], dtype=np.int64)
    check_rows(w, res, rows, 8, layout)


def test_2048_short_requests(dev):
    lens = (mi.u64(901, 1, 2048) % np.uint64(700)).astype(np.int64) + 1
    w = mi.build_workload("many", 2048, 1, 16, lens, 4, "interleaved", "bf16", False, seed=901)
    res = run_gpu(w, dev)
    assert res["status"] == 0
    u = mi.u64(902, 2, 40)
    rows = np.unique((u % np.uint64(w.batch * w.num_heads)).astype(np.int64))
    check_rows(w, res, rows, 4, "interleaved")
    # requests shorter than the shard count leave whole shards empty
    lsep = res["lse_partial"].cpu().numpy().reshape(4, 2048, 16)
    for b in np.where(lens < 4)[0][:8]:
        for s in range(int(lens[b]), 4):
            assert np.all(np.isneginf(lsep[s, b]))


def test_128_heads_nine_query_tokens(dev):
    lens = [5000, 9, 130]
    w = mi.build_workload("h128", 3, 9, 128, lens, 2, "contiguous", "bf16", True, seed=903,
                          poison=True)
    res = run_gpu(w, dev)
    assert res["status"] == 0
    R = 3 * 9 * 128
    u = mi.u64(904, 3, 48)
    rows = np.unique(np.concatenate([[0, R - 1, 9 * 128, 9 * 128 - 1],
                                     (u % np.uint64(R)).astype(np.int64)]))
    check_rows(w, res, rows, 2, "contiguous")
