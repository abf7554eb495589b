"""GPU parity at the full benchmark sizes, in the launch configuration the
benchmark times.  The oracle computes sampled query rows one by one: the
longest and shortest requests plus seeded random ones, every query position
of the causal verify step at its ends, and the per-shard partials of those
rows for every shard.
"""
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


def sample_rows(w, n_random=10, seed=0):
    B, q, H = w.batch, w.q_len, w.num_heads
    u = mi.u64(1000 + seed, 77, 3 * n_random)
    bs = [int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens))]
    bs += [int(x % B) for x in u[:n_random]]
    rows = []
    for k, b in enumerate(bs):
        h = int(u[n_random + (k % n_random)] % H)
        i_list = [0, q - 1] if q > 1 else [0]
        for i in i_list:
            rows.append((b * q + i) * H + h)
    return np.unique(np.array(rows, dtype=np.int64))


def check_sampled(w, res, rows, N, layout):
    R = w.batch * w.q_len * w.num_heads
    out = bf16_to_np(res["out"]).reshape(R, 512)[rows]
    lse = res["lse"].cpu().numpy().reshape(R)[rows]
    ref, ref_lse = oracle.attend(w, shard=-1, rows=rows)
    check_close(out, ref, TOL_OUT, "out", rel=REL_OUT)
    check_close(lse, ref_lse, TOL_LSE, "lse")
    part = res["partial"].cpu().numpy().reshape(N, R, 512)
    lsep = res["lse_partial"].cpu().numpy().reshape(N, R)
    for s in range(N):
        po, pl = oracle.attend(w, shard=s, num_shards=N, layout=layout, rows=rows)
        check_close(part[s][rows], po, TOL_OUT, f"partial {s}", rel=REL_OUT)
        check_close(lsep[s][rows], pl, TOL_LSE, f"lse_partial {s}")
    if w.w_uv is not None:
        y = bf16_to_np(res["y"]).reshape(R, 128)[rows]
        ref_y = oracle.project_wuv(ref, (rows % w.num_heads).astype(np.int32), w.w_uv)
        check_close(y, ref_y, TOL_OUT, "y", rel=REL_OUT)


def test_config1_tiny_all_rows(dev):
    w = mi.config_workload(1)
    res = run_gpu(w, dev)
    assert res["status"] == 0
    rows = np.arange(w.batch * w.q_len * w.num_heads, dtype=np.int64)
    check_sampled(w, res, rows, w.num_shards, w.layout)


def test_config2_bimodal_agentic(dev):
    w = mi.config_workload(2)
    res = run_gpu(w, dev)
    assert res["status"] == 0
    check_sampled(w, res, sample_rows(w, seed=2), w.num_shards, w.layout)


@pytest.fixture(scope="module")
def cfg3():
    return mi.config_workload(3)


@pytest.mark.parametrize("N", [1, 2, 4, 8])
@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
def test_config3_shard_sweep(dev, cfg3, N, layout):
    res = run_gpu(cfg3, dev, num_shards=N, layout=layout)
    assert res["status"] == 0
    check_sampled(cfg3, res, sample_rows(cfg3, n_random=6, seed=3 + N), N, layout)


def test_config4_spec_verify(dev):
    w = mi.config_workload(4)
    res = run_gpu(w, dev)
    assert res["status"] == 0
    check_sampled(w, res, sample_rows(w, seed=4), w.num_shards, w.layout)


def test_config5_longtail_fp8_fused_wuv(dev):
    w = mi.config_workload(5)
    res = run_gpu(w, dev)
    assert res["status"] == 0
    check_sampled(w, res, sample_rows(w, n_random=6, seed=5), w.num_shards, w.layout)
