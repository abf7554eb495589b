"""GPU parity at the full benchmark sizes, in the launch configuration the
benchmark times.  The oracle computes sampled query rows one by one: the
longest and shortest requests plus seeded random ones, every query position
of the causal verify step at its ends, one row of every work unit that the
device's own work plan (read back from the workspace) splits across CTAs --
so every split piece, boundary pieces included, is checked -- and the
per-shard partials of those rows for every shard.  The whole decode step
(mla_decode_step, the call the benchmark times) is checked on the same rows.
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


def split_unit_rows(w, workspace, n_out, seed=0):
    """One seeded row of every work unit the device's plan splits across
    CTAs.  The workspace starts with the plan's header (error word, total
    positions, positions per CTA, grid, units, positions charged per unit)
    and, 256 bytes in, the exclusive prefix of work positions over units."""
    ws = workspace.cpu().numpy()
    hdr = ws[:256].view(np.int32)
    per, U, cost = int(hdr[2]), int(hdr[4]), int(hdr[5])
    prefix = ws[256:256 + 4 * (U + 1)].view(np.int32)
    R = w.q_len * w.num_heads
    G = (R + 63) // 64
    u64 = mi.u64(2000 + seed, 78, U)
    rows = []
    for u in range(U):
        if prefix[u + 1] == prefix[u]:
            continue
        us, ue = prefix[u] + cost, prefix[u + 1]
        if us // per == (ue - 1) // per:
            continue
        g = u % G
        b = u // (G * n_out)
        nrow = min(64, R - 64 * g)
        rows.append(b * R + 64 * g + int(u64[u] % nrow))
    return np.array(sorted(set(rows)), dtype=np.int64)


def run_step(w, dev):
    import torch
    import sequence_sharded_mla_gb300 as mla
    from _helpers import to_device
    t = to_device(w, dev)
    out, lse, ws = mla.mla_decode_step(t["q"], t["kv"], t["block_table"], t["seq_lens"],
                                       w.num_shards, w.layout, kv_scale=t["kv_scale"],
                                       causal=w.causal, softmax_scale=w.softmax_scale,
                                       w_uv=t["w_uv"])
    torch.cuda.synchronize()
    assert mla.mla_get_device_error(ws) == 0
    return out, lse, ws


def check_step(w, dev, rows):
    """The whole decode step on the sampled rows and one row of every unit
    its own plan splits."""
    out, lse, ws = run_step(w, dev)
    rows = np.union1d(rows, split_unit_rows(w, ws, w.num_shards, seed=7))
    R = w.batch * w.q_len * w.num_heads
    ref, ref_lse = oracle.attend(w, shard=-1, rows=rows)
    check_close(lse.cpu().numpy().reshape(R)[rows], ref_lse, TOL_LSE, "step lse")
    if w.w_uv is not None:
        ref_y = oracle.project_wuv(ref, (rows % w.num_heads).astype(np.int32), w.w_uv)
        check_close(bf16_to_np(out).reshape(R, 128)[rows], ref_y, TOL_OUT, "step y",
                    rel=REL_OUT)
    else:
        check_close(bf16_to_np(out).reshape(R, 512)[rows], ref, TOL_OUT, "step out",
                    rel=REL_OUT)
    return len(rows)


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
    rows = np.union1d(sample_rows(w, seed=2),
                      split_unit_rows(w, res["workspace"], w.num_shards, seed=2))
    check_sampled(w, res, rows, w.num_shards, w.layout)


@pytest.mark.parametrize("cfg", [2, 4, 5, "4+wuv"])
def test_decode_step_full_size(dev, cfg):
    """cfg "4+wuv": the q_len-9 batch with a W_UV projection, 144 query rows
    per head, which runs on the tensor cores after the combine."""
    if cfg == "4+wuv":
        w = mi.config_workload(4, with_w_uv=True)
        cfg = 4
    else:
        w = mi.config_workload(cfg)
    n = check_step(w, dev, sample_rows(w, n_random=6, seed=20 + cfg))
    assert n >= 8


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
    rows = np.union1d(sample_rows(w, n_random=6, seed=5),
                      split_unit_rows(w, res["workspace"], w.num_shards, seed=5))
    check_sampled(w, res, rows, w.num_shards, w.layout)
