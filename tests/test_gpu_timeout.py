"""Bounded device waits: a wait that runs out is reported, not hung on.

Every wait of the partial-attention kernels has a time limit.  Here the
kernels are told never to load the query rows of each CTA's first piece (a
testing hook), so the waits for them can only run out, after a budget set to
1 ms.  The call must still return, the error word must read
MLA_ERR_TIMEOUT, and the next ordinary call on the same stream must match the
oracle: the aborted kernel let its own copies drain and freed its tensor
memory, and the next launch re-initialises its barriers.  Nothing here
faults, traps or spins without a limit: the failure is a wait on a barrier
that nothing completes, under a short time limit.
"""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from _helpers import REL_OUT, TOL_LSE, TOL_OUT, check_close, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_wait_budget_runs_out_and_next_call_is_clean(kv_dtype):
    import torch
    import sequence_sharded_mla_gb300 as mla
    dev = torch.device("cuda:0")
    w = mi.build_workload("timeout", 2, 1, 16, [300, 4000], 2, "interleaved", kv_dtype, False,
                          seed=950, kv_sigma=1.0 if kv_dtype == "fp8" else 0.5)
    t = to_device(w, dev)
    try:
        mla.mla_set_wait_budget_ns(1_000_000)
        mla.mla_set_withhold_query(True)
        _, _, ws = mla.mla_decode_partial(t["q"], t["kv"], t["block_table"], t["seq_lens"], 2,
                                          "interleaved", kv_scale=t["kv_scale"])
        torch.cuda.synchronize()
        assert mla.mla_get_device_error(ws) == -4          # MLA_ERR_TIMEOUT
        assert mla.mla_get_device_error(ws) == 0           # read clears it
    finally:
        mla.mla_set_withhold_query(False)
        mla.mla_set_wait_budget_ns(0)
    rows = w.batch * w.q_len * w.num_heads
    for _ in range(2):
        part, lse, ws = mla.mla_decode_partial(t["q"], t["kv"], t["block_table"], t["seq_lens"],
                                               2, "interleaved", kv_scale=t["kv_scale"],
                                               workspace=ws)
        torch.cuda.synchronize()
        assert mla.mla_get_device_error(ws) == 0
        got = part.cpu().numpy().reshape(2, rows, 512)
        got_lse = lse.cpu().numpy().reshape(2, rows)
        for s in range(2):
            ro, rl = oracle.attend(w, shard=s, num_shards=2, layout="interleaved")
            check_close(got[s], ro, TOL_OUT, f"shard {s}", rel=REL_OUT)
            check_close(got_lse[s], rl, TOL_LSE, f"lse shard {s}")
