"""Pins of the GQA oracle (the grouped-query backend of "Decode Context
Parallelism", section 5.4: KV heads broadcast over groups of query heads,
the cache split along the sequence) against things other than itself."""
from decimal import Decimal, getcontext

import numpy as np
import pytest

import mla_inputs as mi
import oracle as orc


def _bf16(bits):
    return float(mi.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0])


def small(seed, B=2, q_len=1, H=4, Hkv=2, D=16, lens=(37, 64), N=2, layout="interleaved",
          causal=False, poison=False):
    return mi.build_gqa_workload("gqa", B, q_len, H, Hkv, D, list(lens), N, layout, causal,
                                 seed, poison=poison)


def brute_force_row(w, b, i, h):
    """One query row in Decimal arithmetic from the definition, with its own
    page lookup and its own head-to-KV-head mapping."""
    getcontext().prec = 50
    L = int(w.seq_lens[b])
    D = w.head_dim
    kh = h // (w.num_heads // w.num_kv_heads)
    q = [Decimal(_bf16(x)) for x in w.q[b, i, h]]
    scale = Decimal(1) / Decimal(D).sqrt()
    num = [Decimal(0)] * D
    den = Decimal(0)
    for t in range(L):
        if w.causal and t > L - w.q_len + i:
            continue
        page = int(w.block_table[b, t // 64])
        k = [Decimal(_bf16(x)) for x in w.k_cache[page, t % 64, kh]]
        v = [Decimal(_bf16(x)) for x in w.v_cache[page, t % 64, kh]]
        e = (sum(a * c for a, c in zip(q, k)) * scale).exp()
        den += e
        for c in range(D):
            num[c] += e * v[c]
    return np.array([float(x / den) for x in num]), float(den.ln())


@pytest.mark.parametrize("seed,H,Hkv,q_len,causal", [(21, 4, 2, 1, False), (22, 4, 1, 2, True),
                                                     (23, 6, 3, 1, False)])
def test_brute_force_matches_oracle(seed, H, Hkv, q_len, causal):
    w = small(seed, H=H, Hkv=Hkv, q_len=q_len, lens=(40, 70), causal=causal)
    out, lse = orc.gqa_attend(w, shard=-1)
    for b in range(w.batch):
        for i in range(q_len):
            for h in range(H):
                r = (b * q_len + i) * H + h
                o, l = brute_force_row(w, b, i, h)
                assert np.allclose(out[r], o, rtol=1e-12, atol=1e-13)
                assert abs(lse[r] - l) < 1e-12


def test_kv_heads_are_broadcast_over_consecutive_query_heads():
    """Query head h with KV head h // (H / Hkv) equals single-head attention
    over a cache that holds only that KV head (built here by slicing)."""
    w = small(31, B=2, H=8, Hkv=2, D=32, lens=(100, 33))
    out, lse = orc.gqa_attend(w, shard=-1)
    G = 4
    for h in range(8):
        kh = h // G
        w1 = mi.GqaWorkload("one", 2, 1, 1, 1, 32, w.seq_lens, 1, "interleaved", False, 0,
                            q=np.ascontiguousarray(w.q[:, :, h:h + 1]),
                            k_cache=np.ascontiguousarray(w.k_cache[:, :, kh:kh + 1]),
                            v_cache=np.ascontiguousarray(w.v_cache[:, :, kh:kh + 1]),
                            block_table=w.block_table, softmax_scale=w.softmax_scale)
        o1, l1 = orc.gqa_attend(w1, shard=-1)
        for b in range(2):
            assert np.array_equal(out[b * 8 + h], o1[b])
            assert lse[b * 8 + h] == l1[b]


def test_single_token_returns_its_value_row():
    w = small(32, B=1, H=4, Hkv=2, D=16, lens=(1,))
    out, lse = orc.gqa_attend(w, shard=-1)
    page = int(w.block_table[0, 0])
    for h in range(4):
        v = mi.bf16_bits_to_f32(w.v_cache[page, 0, h // 2]).astype(np.float64)
        assert np.array_equal(out[h], v)


def test_identical_keys_give_the_mean_of_values():
    w = small(33, B=1, H=2, Hkv=1, D=16, lens=(50,))
    w.k_cache[:] = w.k_cache[int(w.block_table[0, 0]), 0]
    out, lse = orc.gqa_attend(w, shard=-1)
    pages = [int(w.block_table[0, t // 64]) for t in range(50)]
    vals = np.stack([mi.bf16_bits_to_f32(w.v_cache[p, t % 64, 0]) for t, p in enumerate(pages)])
    assert np.allclose(out[0], vals.astype(np.float64).mean(axis=0), rtol=0, atol=1e-12)
    q = mi.bf16_bits_to_f32(w.q[0, 0, 0]).astype(np.float64)
    k = mi.bf16_bits_to_f32(w.k_cache[pages[0], 0, 0]).astype(np.float64)
    s = float(q @ k) * w.softmax_scale
    assert abs(lse[0] - (s + np.log(50))) < 1e-10


@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
@pytest.mark.parametrize("N", [1, 2, 3, 5])
def test_sharded_then_merged_equals_unsharded(layout, N):
    w = small(34, B=3, q_len=2, H=4, Hkv=2, D=16, lens=(130, 7, 64), causal=True)
    ref, ref_lse = orc.gqa_attend(w, shard=-1)
    parts = [orc.gqa_attend(w, shard=s, num_shards=N, layout=layout) for s in range(N)]
    o, l = orc.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(o, ref, rtol=0, atol=1e-12)
    assert np.allclose(l, ref_lse, rtol=0, atol=1e-12)


def test_page_permutation_and_poisoned_rows():
    w = small(35, B=2, H=4, Hkv=2, D=16, lens=(90, 10), poison=True)
    out, lse = orc.gqa_attend(w, shard=-1)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    perm = np.random.default_rng(0).permutation(w.num_pages)
    inv = np.argsort(perm)
    w2 = mi.GqaWorkload("perm", 2, 1, 4, 2, 16, w.seq_lens, 2, "interleaved", False, 0, q=w.q,
                        k_cache=np.ascontiguousarray(w.k_cache[perm]),
                        v_cache=np.ascontiguousarray(w.v_cache[perm]),
                        block_table=np.where(w.block_table >= 0, inv[np.maximum(w.block_table, 0)],
                                             -1).astype(np.int32),
                        softmax_scale=w.softmax_scale)
    o2, l2 = orc.gqa_attend(w2, shard=-1)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_causal_row_equals_shorter_decode():
    w = small(36, B=1, q_len=3, H=2, Hkv=1, D=16, lens=(80,), causal=True)
    out, lse = orc.gqa_attend(w, shard=-1)
    for i in range(3):
        w1 = mi.GqaWorkload("q1", 1, 1, 2, 1, 16, np.array([80 - 2 + i], dtype=np.int32), 1,
                            "interleaved", False, 0, q=np.ascontiguousarray(w.q[:, i:i + 1]),
                            k_cache=w.k_cache, v_cache=w.v_cache, block_table=w.block_table,
                            softmax_scale=w.softmax_scale)
        o1, l1 = orc.gqa_attend(w1, shard=-1)
        assert np.array_equal(out[i * 2:(i + 1) * 2], o1) and np.array_equal(lse[i * 2:(i + 1) * 2], l1)
