"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every output element: per-shard partials and LSEs, the
LSE-combined bf16 output and LSE, and the fused W_UV projection.  They span
several 64-token tiles with ragged tails, empty shards, both shard layouts,
N = 1..8, 16..64 heads, q_len 1/2/9 (causal), bf16 and fp8 caches and
NaN-poisoned unused cache rows.  Full-size configurations are checked on
sampled query rows in test_gpu_configs.py.
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


def compare_all(w, dev, layout=None, N=None):
    N = w.num_shards if N is None else N
    lay = w.layout if layout is None else layout
    res = run_gpu(w, dev, num_shards=N, layout=lay)
    assert res["status"] == 0, res["status"]
    rows = w.batch * w.q_len * w.num_heads
    part = res["partial"].cpu().numpy().reshape(N, rows, 512)
    lsep = res["lse_partial"].cpu().numpy().reshape(N, rows)
    for s in range(N):
        ro, rl = oracle.attend(w, shard=s, num_shards=N, layout=lay)
        check_close(part[s], ro, TOL_OUT, f"partial shard {s}", rel=REL_OUT)
        check_close(lsep[s], rl, TOL_LSE, f"lse_partial shard {s}")
    ref, ref_lse, ref_y = oracle.reference_step(w)
    check_close(bf16_to_np(res["out"]).reshape(rows, 512), ref, TOL_OUT, "out", rel=REL_OUT)
    check_close(res["lse"].cpu().numpy().reshape(rows), ref_lse, TOL_LSE, "lse")
    if ref_y is not None:
        check_close(bf16_to_np(res["y"]).reshape(rows, 128), ref_y, TOL_OUT, "y", rel=REL_OUT)
    return res


@pytest.mark.parametrize("H", [16, 32, 64])
@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
def test_ragged_lengths(dev, H, layout):
    lens = [1, 2, 63, 64, 65, 1000, 333]
    w = mi.build_workload("ragged", len(lens), 1, H, lens, 2, layout, "bf16", False,
                          seed=100 + H, poison=True, extra_pages=3)
    compare_all(w, dev)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
def test_shard_counts(dev, N, layout):
    """Every shard count, both layouts.  Interleaved shard counts that do not
    divide the page size (3, 5, 6, 7) take each page's rows of a shard as a
    padded run of slots, loaded 8 rows at a time with the rows past the
    page's end outside the load."""
    lens = [5, 700, 2049, 130]
    w = mi.build_workload("shards", len(lens), 1, 32, lens, N, layout, "bf16", False,
                          seed=200 + N, poison=True, extra_pages=2)
    compare_all(w, dev)


@pytest.mark.parametrize("N", [3, 5, 6, 7])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_interleaved_shard_counts_not_dividing_the_page(dev, N, kv_dtype):
    """Long contexts (split units), causal verify rows, a context that ends
    in the pool's last page, and NaN-poisoned rows everywhere outside the
    contexts: interleaved shards whose count does not divide 64."""
    lens = [1, 64, 65, 4000, 9001]
    w = mi.build_workload("padded", len(lens), 2, 16, lens, N, "interleaved", kv_dtype, True,
                          seed=260 + N, poison=True, kv_sigma=1.0 if kv_dtype == "fp8" else 0.5)
    # make the last request's last page the pool's last page: swap the two
    # physical pages' contents (poison included) along with their entries
    last = w.kv.shape[0] - 1
    b, k = len(lens) - 1, (lens[-1] - 1) // 64
    other = int(w.block_table[b, k])
    if other != last:
        j = tuple(np.argwhere(w.block_table == last)[0])
        w.block_table[j], w.block_table[b, k] = other, last
        w.kv[[other, last]] = w.kv[[last, other]]
        if w.kv_scale is not None:
            w.kv_scale[[other, last]] = w.kv_scale[[last, other]]
    assert int(w.block_table[b, k]) == last
    compare_all(w, dev)


@pytest.mark.parametrize("q_len", [2, 9])
@pytest.mark.parametrize("H", [16, 64])
def test_causal_verify(dev, q_len, H):
    lens = [8000 // 8, 130, 9, 64]
    w = mi.build_workload("verify", len(lens), q_len, H, lens, 2, "interleaved", "bf16", True,
                          seed=300 + q_len + H, poison=True)
    compare_all(w, dev)


def test_causal_context_shorter_than_query(dev):
    """Rows that see no token at all give lse = -inf and a zero output."""
    w = mi.build_workload("tiny", 2, 9, 16, [5, 1], 2, "contiguous", "bf16", True, seed=310)
    compare_all(w, dev)


def test_empty_shards(dev):
    w = mi.build_workload("empty", 3, 1, 16, [1, 3, 7], 8, "interleaved", "bf16", False, seed=320)
    compare_all(w, dev)
    w = mi.build_workload("empty", 3, 1, 16, [1, 3, 7], 8, "contiguous", "bf16", False, seed=321)
    compare_all(w, dev)


def test_single_shard_call_matches_all_shards(dev):
    """A per-shard call (the per-GPU call of a multi-GPU deployment) gives the
    same partials as the all-shards call.  The two calls split the work list
    at different points, and each split piece rounds its probabilities to
    bf16 against its own running maximum, so the two agree to the bf16
    probability rounding bound (REL_OUT), not bitwise."""
    w = mi.build_workload("one", 3, 1, 32, [100, 1000, 64], 4, "interleaved", "bf16", False,
                          seed=330)
    full = run_gpu(w, dev)
    for s in range(4):
        one = run_gpu(w, dev, shard_id=s)
        assert one["status"] == 0
        a = one["partial"].cpu().numpy()[0]
        b = full["partial"].cpu().numpy()[s]
        check_close(a, b, TOL_OUT, f"shard {s}", rel=REL_OUT)
        la = one["lse_partial"].cpu().numpy()[0]
        lb = full["lse_partial"].cpu().numpy()[s]
        check_close(la, lb, TOL_LSE, f"lse shard {s}")


def test_deterministic(dev):
    w = mi.build_workload("det", 4, 1, 64, [5000, 70, 20000, 1], 4, "interleaved", "bf16", False,
                          seed=340)
    a = run_gpu(w, dev)
    b = run_gpu(w, dev)
    assert np.array_equal(a["partial"].cpu().numpy(), b["partial"].cpu().numpy())
    import torch
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["lse"], b["lse"])


def test_fused_wuv_small(dev):
    w = mi.build_workload("wuv", 3, 1, 32, [100, 3000, 17], 4, "interleaved", "bf16", False,
                          seed=350, with_w_uv=True)
    compare_all(w, dev)


def test_bad_block_table_entry_reports_bounds_error(dev):
    import sequence_sharded_mla_gb300 as mla
    w = mi.build_workload("bad", 2, 1, 16, [200, 64], 2, "interleaved", "bf16", False, seed=360)
    w.block_table[0, 2] = w.num_pages + 100
    res = run_gpu(w, dev)
    assert res["status"] == -5          # MLA_ERR_DEVICE_BOUNDS
    assert mla.mla_get_device_error(res["workspace"]) == 0   # read clears it
    assert np.all(np.isfinite(res["partial"].cpu().numpy()))


def test_invalid_arguments_rejected_before_launch(dev):
    import torch
    import sequence_sharded_mla_gb300 as mla
    w = mi.build_workload("inv", 1, 1, 16, [64], 2, "interleaved", "bf16", False, seed=370)
    from _helpers import to_device
    t = to_device(w, dev)
    with pytest.raises(mla.MLAError) as e:
        mla.mla_decode_partial(t["q"], t["kv"], t["block_table"], t["seq_lens"], 9)
    assert e.value.status == -1
    q20 = torch.zeros((1, 1, 20, 576), dtype=torch.bfloat16, device=dev)
    with pytest.raises(mla.MLAError) as e:
        mla.mla_decode_partial(q20, t["kv"], t["block_table"], t["seq_lens"], 2)
    assert e.value.status == -2          # heads must be a multiple of 16
    small_ws = torch.empty((64,), dtype=torch.uint8, device=dev)
    with pytest.raises(mla.MLAError) as e:
        mla.mla_decode_partial(t["q"], t["kv"], t["block_table"], t["seq_lens"], 2,
                               workspace=small_ws)
    assert e.value.status == -6


@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
@pytest.mark.parametrize("N", [1, 2, 8])
def test_fp8_cache(dev, layout, N):
    """fp8 e4m3 cache with one fp32 scale per token; unused rows and pages
    carry NaN codes and NaN scales."""
    lens = [1, 63, 65, 1000, 4097]
    w = mi.build_workload("fp8", len(lens), 1, 64, lens, N, layout, "fp8", False, seed=400 + N,
                          kv_sigma=1.0, poison=True, extra_pages=2)
    compare_all(w, dev)


def test_fp8_causal_verify_with_wuv(dev):
    w = mi.build_workload("fp8v", 3, 9, 32, [300, 9, 2000], 2, "interleaved", "fp8", True,
                          seed=410, kv_sigma=1.0, poison=True, with_w_uv=True)
    compare_all(w, dev)


def test_fp8_query_of_any_finite_magnitude(dev):
    """With fp8 caches the query enters the tensor cores as a two-term e4m3
    sum under a per-row power-of-two scale.  The cache's scales are divided by
    2^20 and one head's query multiplied by 2^20 (|q| up to ~1e6, beyond fp16),
    another's divided by 2^100: all rows match the oracle."""
    import numpy as np
    w = mi.build_workload("fp8big", 2, 1, 16, [100, 700], 2, "interleaved", "fp8", False,
                          seed=420, kv_sigma=1.0)
    w.kv_scale *= np.float32(2.0 ** -20)

    def shift_exponent(x, k):   # multiply nonzero bf16 patterns by 2^k
        nz = (x & 0x7F80) != 0
        x[nz] = (x[nz].astype(np.int32) + (k << 7)).astype(np.uint16)

    for b in range(2):
        shift_exponent(w.q[b, 0, 3, :], 20)
        shift_exponent(w.q[b, 0, 5, :], -100)
    assert np.max(np.abs(mi.bf16_bits_to_f32(w.q[0, 0, 3, :]))) > 65504.0
    compare_all(w, dev)


def test_fp8_nonfinite_query_is_reported(dev):
    """An inf or NaN query component of a row that attends is reported as
    MLA_ERR_RANGE; a padding row's garbage is not."""
    w = mi.build_workload("fp8inf", 1, 1, 16, [100], 2, "interleaved", "fp8", False, seed=421,
                          kv_sigma=1.0)
    w.q[0, 0, 3, 7] = 0x7F80          # bf16 +inf
    res = run_gpu(w, dev, with_wuv=False)
    assert res["status"] == -7          # MLA_ERR_RANGE
    w.q[0, 0, 3, 7] = 0x7FC0          # bf16 NaN
    res = run_gpu(w, dev, with_wuv=False)
    assert res["status"] == -7
    # the second query slot of the request is padding (q_lens = 1)
    w = mi.build_workload("fp8pad", 1, 2, 16, [100], 2, "interleaved", "fp8", True, seed=422,
                          kv_sigma=1.0, q_lens=[1])
    w.q[0, 1, :, :] = 0x7FC0
    res = run_gpu(w, dev, with_wuv=False)
    assert res["status"] == 0


def test_fp8_token_scales_of_any_magnitude(dev):
    """Token scales multiplied by 2^k, k uniform in [-40, 2] (logits stay of
    order 10, the values span 2^42), some exactly zero and some negative: the
    exponent split of the scales keeps P' inside e4m3 and the normaliser
    exact, so the many near-zero-logit tokens keep their weight."""
    import numpy as np
    w = mi.build_workload("fp8sc", 3, 2, 32, [130, 1000, 4100], 4, "interleaved", "fp8", True,
                          seed=450, kv_sigma=1.0)
    rng = np.random.default_rng(451)
    sc = w.kv_scale.reshape(-1)
    sc *= np.exp2(rng.integers(-40, 3, size=sc.shape)).astype(np.float32)
    sc[rng.random(sc.shape) < 0.02] = 0.0
    neg = rng.random(sc.shape) < 0.05
    sc[neg] = -sc[neg]
    compare_all(w, dev)


def test_fp8_small_query_values_stay_within_tolerance(dev):
    """Tiny query components (sigma 1e-5): the per-row power-of-two scale
    brings them into the e4m3 range before the two-term split."""
    w = mi.build_workload("fp8tiny", 2, 1, 32, [700, 1300], 2, "contiguous", "fp8", False,
                          seed=430, kv_sigma=1.0, q_sigma=1e-5)
    compare_all(w, dev)


@pytest.mark.parametrize("layout,N", [("interleaved", 2), ("interleaved", 3), ("interleaved", 8),
                                      ("contiguous", 3), ("contiguous", 4)])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_local_shard_caches(dev, layout, N, kv_dtype):
    """Each shard computed from a cache that holds only its own positions (the
    layout each GPU of a multi-GPU deployment stores) equals that shard's
    partial over the whole cache, causal verify included; the combine of all
    shards equals unsharded attention."""
    import torch
    import sequence_sharded_mla_gb300 as mla
    lens = [1, 100, 777, 4099]
    w = mi.build_workload("local", len(lens), 2, 32, lens, N, layout, kv_dtype, True,
                          seed=440 + N, kv_sigma=1.0 if kv_dtype == "fp8" else 0.5, poison=True)
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    rows = w.batch * w.q_len * w.num_heads
    parts, lses = [], []
    for s in range(N):
        d = mi.local_shard_cache(w, N, s, layout, seed=s)
        if kv_dtype == "bf16":
            kv = torch.from_numpy(d["kv"].view(np.int16)).view(torch.bfloat16).to(dev)
            sc = None
        else:
            kv = torch.from_numpy(d["kv"]).to(dev)
            sc = torch.from_numpy(d["kv_scale"]).to(dev)
        bt = torch.from_numpy(d["block_table"]).to(dev)
        part, lse, ws = mla.mla_decode_partial(q, kv, bt, sl, N, layout + "_local", shard_id=s,
                                               kv_scale=sc, causal=True)
        torch.cuda.synchronize()
        assert mla.mla_get_device_error(ws) == 0
        ref_o, ref_l = oracle.attend(w, shard=s, num_shards=N, layout=layout)
        check_close(part.cpu().numpy().reshape(rows, 512), ref_o, TOL_OUT, f"local shard {s}",
                    rel=REL_OUT)
        check_close(lse.cpu().numpy().reshape(rows), ref_l, TOL_LSE, f"local lse {s}")
        parts.append(part[0])
        lses.append(lse[0])
    out, lse_out = mla.mla_shard_combine(torch.stack(parts), torch.stack(lses), causal=True)
    torch.cuda.synchronize()
    ref, ref_lse, _ = oracle.reference_step(w)
    check_close(bf16_to_np(out).reshape(rows, 512), ref, TOL_OUT, "out", rel=REL_OUT)
    check_close(lse_out.cpu().numpy().reshape(rows), ref_lse, TOL_LSE, "lse")


@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
@pytest.mark.parametrize("causal", [True, False])
def test_variable_query_counts(dev, layout, causal):
    """A padded batch of verify steps with different draft counts: rows past
    a request's count are padding (o = 0, lse = -inf); the causal mask uses
    each request's own count.  32 heads x q_len 9 = 288 rows, so groups of
    64 rows end inside requests' padding."""
    lens = [1, 300, 5000, 64, 2222]
    w = mi.build_workload("qlens", len(lens), 9, 32, lens, 2, layout, "bf16", causal,
                          seed=460, poison=True, q_lens=[1, 9, 4, 2, 7])
    compare_all(w, dev)


def test_variable_query_counts_fp8_local_and_wuv(dev):
    import torch
    import sequence_sharded_mla_gb300 as mla
    lens = [700, 65, 3000]
    w = mi.build_workload("qlens8", len(lens), 4, 48, lens, 4, "interleaved", "fp8", True,
                          seed=470, kv_sigma=1.0, with_w_uv=True, q_lens=[4, 1, 3])
    compare_all(w, dev)
    from _helpers import to_device
    t = to_device(w, dev)
    rows = w.batch * w.q_len * w.num_heads
    for s in range(3):
        d = mi.local_shard_cache(w, 3, s, "interleaved", seed=s)
        part, lse, ws = mla.mla_decode_partial(
            t["q"], torch.from_numpy(d["kv"]).to(dev), torch.from_numpy(d["block_table"]).to(dev),
            t["seq_lens"], 3, "interleaved_local", shard_id=s,
            kv_scale=torch.from_numpy(d["kv_scale"]).to(dev), causal=True, q_lens=t["q_lens"])
        torch.cuda.synchronize()
        assert mla.mla_get_device_error(ws) == 0
        ro, rl = oracle.attend(w, shard=s, num_shards=3, layout="interleaved")
        check_close(part.cpu().numpy().reshape(rows, 512), ro, TOL_OUT, f"shard {s}", rel=REL_OUT)
        check_close(lse.cpu().numpy().reshape(rows), rl, TOL_LSE, f"lse {s}")


def test_query_count_out_of_range_is_reported(dev):
    import torch
    import sequence_sharded_mla_gb300 as mla
    w = mi.build_workload("qbad", 2, 3, 16, [100, 200], 2, "interleaved", "bf16", True, seed=480,
                          q_lens=[3, 4])
    res = run_gpu(w, dev)
    assert res["status"] == -1           # MLA_ERR_INVALID: 4 > q_len
    assert mla.mla_get_device_error(res["workspace"]) == 0
    w.q_lens = np.array([0, 2], dtype=np.int32)
    res = run_gpu(w, dev)
    assert res["status"] == -1
