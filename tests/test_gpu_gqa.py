"""GPU parity of the grouped-query backend (C ABI gqa_* calls) against the
fp64 GQA oracle: every element of small ragged cases over KV-head counts,
group sizes, shard counts, both layouts and causal verify; sampled rows of a
full-size batch."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from _helpers import REL_OUT, TOL_LSE, TOL_OUT, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    return torch.device("cuda:0")


def to_dev(w, dev):
    import torch
    f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return (f(w.q), f(w.k_cache), f(w.v_cache), torch.from_numpy(w.block_table).to(dev),
            torch.from_numpy(w.seq_lens).to(dev))


def run(w, dev, N=None, layout=None, shard_id=-1):
    import torch
    import sequence_sharded_mla_gb300 as mla
    q, k, v, bt, sl = to_dev(w, dev)
    N = w.num_shards if N is None else N
    part, lse, ws = mla.gqa_decode_partial(q, k, v, bt, sl, N, layout or w.layout,
                                           shard_id=shard_id, causal=w.causal)
    out = lse_out = None
    if shard_id == -1:
        out, lse_out = mla.gqa_shard_combine(part, lse)
    torch.cuda.synchronize()
    return part, lse, out, lse_out, mla.mla_get_device_error(ws)


def compare_all(w, dev, N=None, layout=None):
    N = w.num_shards if N is None else N
    lay = layout or w.layout
    part, lse, out, lse_out, status = run(w, dev, N, lay)
    assert status == 0
    rows = w.batch * w.q_len * w.num_heads
    D = w.head_dim
    part = part.cpu().numpy().reshape(N, rows, D)
    lse = lse.cpu().numpy().reshape(N, rows)
    for s in range(N):
        ro, rl = oracle.gqa_attend(w, shard=s, num_shards=N, layout=lay)
        check_close(part[s], ro, TOL_OUT, f"partial {s}", rel=REL_OUT)
        check_close(lse[s], rl, TOL_LSE, f"lse {s}")
    ref, ref_lse = oracle.gqa_attend(w, shard=-1)
    check_close(out.float().cpu().numpy().reshape(rows, D), ref, TOL_OUT, "out", rel=REL_OUT)
    check_close(lse_out.cpu().numpy().reshape(rows), ref_lse, TOL_LSE, "lse")


@pytest.mark.parametrize("H,Hkv", [(8, 8), (16, 8), (16, 4), (32, 4), (64, 4), (64, 1)])
def test_group_sizes(dev, H, Hkv):
    lens = [1, 63, 65, 700, 3001]
    w = mi.build_gqa_workload("gqa", len(lens), 1, H, Hkv, 128, lens, 2, "interleaved", False,
                              seed=700 + H + Hkv, poison=True, extra_pages=2)
    compare_all(w, dev)


@pytest.mark.parametrize("N,layout", [(1, "interleaved"), (4, "interleaved"), (8, "interleaved"),
                                      (3, "contiguous"), (5, "contiguous")])
def test_shard_counts_and_layouts(dev, N, layout):
    lens = [5, 400, 2049, 130]
    w = mi.build_gqa_workload("gqa-n", len(lens), 1, 32, 8, 128, lens, N, layout, False,
                              seed=720 + N, poison=True)
    compare_all(w, dev)


@pytest.mark.parametrize("q_len,H,Hkv", [(3, 16, 4), (9, 64, 8), (5, 32, 1)])
def test_causal_verify(dev, q_len, H, Hkv):
    """q_len x group heads beyond 64 rows spread over several row groups."""
    lens = [1000, 70, 9]
    w = mi.build_gqa_workload("gqa-c", len(lens), q_len, H, Hkv, 128, lens, 2, "interleaved",
                              True, seed=740 + q_len, poison=True)
    compare_all(w, dev)


def test_single_shard_call_matches_all_shards(dev):
    lens = [300, 1200]
    w = mi.build_gqa_workload("gqa-1", 2, 1, 16, 2, 128, lens, 4, "interleaved", False, seed=760)
    part_all, lse_all, _, _, st = run(w, dev)
    assert st == 0
    for s in range(4):
        p1, l1, _, _, st = run(w, dev, shard_id=s)
        assert st == 0
        # the two calls split the work differently over CTAs, so P is rounded
        # to bf16 at different running maxima: equal within the parity bound
        check_close(p1[0].cpu().numpy().reshape(-1, 128), part_all[s].cpu().numpy().reshape(-1, 128),
                    TOL_OUT, f"shard {s}", rel=REL_OUT)
        check_close(l1[0].cpu().numpy().ravel(), lse_all[s].cpu().numpy().ravel(), TOL_LSE,
                    f"lse {s}")


def test_unsupported_shapes_are_refused(dev):
    import torch
    import sequence_sharded_mla_gb300 as mla
    w = mi.build_gqa_workload("gqa-bad", 1, 1, 12, 4, 128, [100], 2, "interleaved", False, seed=770)
    with pytest.raises(mla.MLAError) as e:       # groups of 3 heads
        run(w, dev)
    assert e.value.status == -2
    w = mi.build_gqa_workload("gqa-bad2", 1, 1, 8, 2, 64, [100], 2, "interleaved", False, seed=771)
    with pytest.raises(mla.MLAError) as e:       # head width 64
        run(w, dev)
    assert e.value.status == -2


def test_full_size_agentic_batch_sampled_rows(dev):
    """32 requests of the bimodal agentic length mix, 64 query heads over 4 KV
    heads of width 128, 2 interleaved shards; sampled rows of every shard."""
    w = mi.config_gqa_workload()
    part, lse, out, lse_out, st = run(w, dev)
    assert st == 0
    rows_total = w.batch * w.q_len * w.num_heads
    u = mi.u64(880, 77, 24)
    rows = np.unique(np.concatenate([
        [int(np.argmax(w.seq_lens)) * w.num_heads + h for h in (0, 63)],
        [int(np.argmin(w.seq_lens)) * w.num_heads + 5],
        (u % rows_total).astype(np.int64)]))
    D = w.head_dim
    N = w.num_shards
    part = part.cpu().numpy().reshape(N, rows_total, D)
    lse = lse.cpu().numpy().reshape(N, rows_total)
    for s in range(N):
        ro, rl = oracle.gqa_attend(w, shard=s, rows=rows)
        check_close(part[s][rows], ro, TOL_OUT, f"partial {s}", rel=REL_OUT)
        check_close(lse[s][rows], rl, TOL_LSE, f"lse {s}")
    ref, ref_lse = oracle.gqa_attend(w, shard=-1, rows=rows)
    check_close(out.float().cpu().numpy().reshape(rows_total, D)[rows], ref, TOL_OUT, "out",
                rel=REL_OUT)
    check_close(lse_out.cpu().numpy().reshape(rows_total)[rows], ref_lse, TOL_LSE, "lse")
