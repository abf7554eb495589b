"""Pins for the fp64 oracle: checks against things other than itself.

Each test fixes the oracle to a fact the pages or mathematics fix:
brute force in 50-digit decimal arithmetic without max subtraction, closed
forms, the LSE-merge identity, the page's own contiguous-sharding example,
gather invariances, the causal verify reading, and the e4m3 code table.
"""
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

import mla_inputs as mi
import oracle as orc

HERE = os.path.dirname(os.path.abspath(__file__))


def small(seed, B=2, q_len=1, H=2, lens=(37, 64), N=2, layout="interleaved", causal=False,
          kv_dtype="bf16", extra_pages=0, poison=False, kv_sigma=0.5):
    return mi.build_workload("small", B, q_len, H, list(lens), N, layout, kv_dtype, causal,
                             seed, kv_sigma=kv_sigma, extra_pages=extra_pages, poison=poison)


def rows_of(w):
    return w.batch * w.q_len * w.num_heads


# --------------------------------------------------------------- brute force
def _bf16(bits):
    return float(mi.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0])


def cache_row_decimal(w, page, row):
    """Row ``row`` of page ``page`` as exact Decimals: bf16 bits decoded, or
    e4m3 codes decoded by the closed form of the format (written out below,
    independent of the oracle's decoder) times the token's own fp32 scale,
    on all 576 entries (one scale per token: latent and rope alike)."""
    if w.kv_dtype == "bf16":
        return [Decimal(_bf16(x)) for x in w.kv[page, row]]
    sc = Decimal(float(w.kv_scale[page, row]))
    return [Decimal(e4m3_closed_form(int(c))) * sc for c in w.kv[page, row]]


def brute_force_row(w, b, i, h):
    """Attention for one query row in Decimal arithmetic, straight from the
    definition: exp of the scaled logits without subtracting a maximum,
    normalised by their sum.  Page lookup written independently here."""
    getcontext().prec = 50
    L = int(w.seq_lens[b])
    q = [Decimal(_bf16(x)) for x in w.q[b, i, h]]
    scale = Decimal(1) / Decimal(192).sqrt()
    num = [Decimal(0)] * 512
    den = Decimal(0)
    for t in range(L):
        if w.causal and t > L - w.q_len + i:
            continue
        page = int(w.block_table[b, t // 64])
        k = cache_row_decimal(w, page, t % 64)
        s = sum(qa * ka for qa, ka in zip(q, k)) * scale
        e = s.exp()
        den += e
        for c in range(512):
            num[c] += e * k[c]
    out = np.array([float(x / den) for x in num])
    return out, float(den.ln())


@pytest.mark.parametrize("seed,lens,q_len,causal", [(11, (1, 64), 1, False),
                                                     (12, (65, 30), 1, False),
                                                     (13, (20, 9), 2, True)])
def test_brute_force_matches_oracle(seed, lens, q_len, causal):
    w = small(seed, lens=lens, q_len=q_len, causal=causal)
    out, lse = orc.attend(w, shard=-1)
    H = w.num_heads
    for b in range(w.batch):
        for i in range(w.q_len):
            for h in range(H):
                r = (b * w.q_len + i) * H + h
                bo, bl = brute_force_row(w, b, i, h)
                assert abs(bl - lse[r]) <= 1e-12 * max(1.0, abs(bl))
                assert np.max(np.abs(bo - out[r])) <= 1e-12 * max(1e-3, np.max(np.abs(bo)))


def spread_token_scales(w, seed):
    """Multiply every token's scale of an fp8 cache by its own factor,
    log-uniform over 2^-2 .. 2^2 and different for every row of a page, so
    that a scale looked up by page, by the wrong row, or applied to only
    part of a row changes the result."""
    u = mi.uniform01(seed, 3, w.kv_scale.size).reshape(w.kv_scale.shape)
    f = np.exp2(-2.0 + 4.0 * u) * (1.0 + (np.arange(64)[None, :] % 5) / 8.0)
    w.kv_scale[...] = (w.kv_scale * f).astype(np.float32)
    return w


@pytest.mark.parametrize("seed,lens,q_len,causal", [(14, (1, 64), 1, False),
                                                     (15, (65, 30), 1, False),
                                                     (16, (20, 9), 2, True)])
def test_brute_force_matches_oracle_fp8(seed, lens, q_len, causal):
    """The fp8 gather: e4m3 code times the token's scale on every entry."""
    w = spread_token_scales(small(seed, lens=lens, q_len=q_len, causal=causal,
                                  kv_dtype="fp8", kv_sigma=1.0), seed)
    assert len(np.unique(w.kv_scale[w.block_table[0, 0]])) > 32
    out, lse = orc.attend(w, shard=-1)
    H = w.num_heads
    for b in range(w.batch):
        for i in range(w.q_len):
            for h in range(H):
                r = (b * w.q_len + i) * H + h
                bo, bl = brute_force_row(w, b, i, h)
                assert abs(bl - lse[r]) <= 1e-12 * max(1.0, abs(bl))
                assert np.max(np.abs(bo - out[r])) <= 1e-12 * max(1e-3, np.max(np.abs(bo)))


# --------------------------------------------------------------- closed forms
def test_single_token_returns_its_value():
    w = small(21, lens=(1, 1))
    out, lse = orc.attend(w, shard=-1)
    for b in range(2):
        page = w.block_table[b, 0]
        v = mi.bf16_bits_to_f32(w.kv[page, 0]).astype(np.float64)
        for h in range(2):
            r = b * 2 + h
            q = mi.bf16_bits_to_f32(w.q[b, 0, h]).astype(np.float64)
            assert np.array_equal(out[r], v[:512])          # out = V_0 exactly
            s0 = float(np.dot(q, v)) / math.sqrt(192.0)
            assert abs(lse[r] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_fp8_single_token_returns_its_scaled_value():
    """A one-token context of an fp8 cache returns that token's dequantised
    latent, code by code times its own scale, and the lse is its logit."""
    w = spread_token_scales(small(23, lens=(1, 1), kv_dtype="fp8", kv_sigma=1.0), 23)
    out, lse = orc.attend(w, shard=-1)
    for b in range(2):
        page = int(w.block_table[b, 0])
        sc = float(w.kv_scale[page, 0])
        v = np.array([e4m3_closed_form(int(c)) for c in w.kv[page, 0]]) * sc
        for h in range(2):
            r = b * 2 + h
            q = mi.bf16_bits_to_f32(w.q[b, 0, h]).astype(np.float64)
            assert np.array_equal(out[r], v[:512])
            s0 = float(np.dot(q, v)) / math.sqrt(192.0)
            assert abs(lse[r] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_fp8_scale_belongs_to_its_token():
    """Scaling one token's scale by 2^k scales its whole dequantised row:
    the same result as a bf16-free fp64 recomputation with that row's
    values multiplied by 2^k, and different from scaling a neighbour."""
    w = spread_token_scales(small(24, B=1, lens=(3,), kv_dtype="fp8", kv_sigma=1.0), 24)
    page = int(w.block_table[0, 0])
    base, base_lse = orc.attend(w, shard=-1)
    w.kv_scale[page, 1] *= 1.5
    o1, l1 = orc.attend(w, shard=-1)
    rows = [np.array([e4m3_closed_form(int(c)) for c in w.kv[page, t]]) * float(w.kv_scale[page, t])
            for t in range(3)]
    K = np.stack(rows)
    for h in range(2):
        q = mi.bf16_bits_to_f32(w.q[0, 0, h]).astype(np.float64)
        s = K @ q / math.sqrt(192.0)
        m = s.max()
        p = np.exp(s - m)
        want = p @ K[:, :512] / p.sum()
        assert np.max(np.abs(o1[h] - want)) <= 1e-12 * max(1.0, np.max(np.abs(want)))
        assert abs(l1[h] - (m + math.log(p.sum()))) <= 1e-12 * max(1.0, abs(m))
    assert not np.allclose(o1, base)


def test_identical_keys_return_mean_of_values():
    """Scores depend only on k_rope when q's latent part is zero; with one
    shared k_rope every token scores the same, so out = mean of c_kv rows
    and lse = s + ln L."""
    w = small(22, lens=(50, 128))
    w.q[:, :, :, :512] = 0
    rope = w.kv[w.block_table[0, 0], 0, 512:].copy()
    w.kv[:, :, 512:] = rope
    out, lse = orc.attend(w, shard=-1)
    ropev = mi.bf16_bits_to_f32(rope).astype(np.float64)
    for b in range(2):
        L = int(w.seq_lens[b])
        rows = [w.kv[w.block_table[b, t // 64], t % 64, :512] for t in range(L)]
        mean = np.mean(mi.bf16_bits_to_f32(np.stack(rows)).astype(np.float64), axis=0)
        for h in range(2):
            r = b * 2 + h
            q = mi.bf16_bits_to_f32(w.q[b, 0, h, 512:]).astype(np.float64)
            s = float(np.dot(q, ropev)) / math.sqrt(192.0)
            assert np.max(np.abs(out[r] - mean)) <= 1e-14
            assert abs(lse[r] - (s + math.log(L))) <= 1e-12 * max(1.0, abs(s) + math.log(L))


# ------------------------------------------------------- sharding and merge
@pytest.mark.parametrize("layout", ["interleaved", "contiguous"])
def test_sharded_then_merged_equals_unsharded(layout):
    w = small(31, B=3, H=2, lens=(1, 7, 200))
    ref, ref_lse = orc.attend(w, shard=-1)
    for N in list(range(1, 9)) + [201]:
        parts = [orc.attend(w, shard=s, num_shards=N, layout=layout) for s in range(N)]
        out, lse = orc.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        assert np.max(np.abs(out - ref)) <= 1e-12, (N, layout)
        assert np.max(np.abs(lse - ref_lse)) <= 1e-12, (N, layout)


def test_shards_partition_tokens():
    """Every token belongs to exactly one shard, in both layouts."""
    for L in (1, 5, 63, 64, 65, 1000):
        for N in range(1, 9):
            for layout in ("interleaved", "contiguous"):
                owners = [orc.token_owner(t, L, N, layout) for t in range(L)]
                assert all(0 <= o < N for o in owners)
                if layout == "interleaved":
                    assert owners == [t % N for t in range(L)]
                else:
                    assert owners == sorted(owners)


def test_contiguous_sharding_matches_page_example():
    path = os.path.join(HERE, "golden", "dcp_contiguous_example.txt")
    lines = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    L, N = map(int, lines[0])
    for t, s in lines[1:]:
        assert orc.token_owner(int(t), L, N, "contiguous") == int(s)


def test_empty_shard_has_minus_inf_lse_and_zero_output():
    w = small(32, lens=(3, 2))
    out, lse = orc.attend(w, shard=4, num_shards=6, layout="interleaved")
    assert np.all(np.isneginf(lse)) and np.all(out == 0)
    out, lse = orc.attend(w, shard=5, num_shards=6, layout="contiguous")
    assert np.all(np.isneginf(lse)) and np.all(out == 0)


def test_lse_merge_matches_textbook_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(5)
    outs = rng.normal(size=(5, 7, 512))
    lses = rng.normal(scale=3, size=(5, 7))
    lses[2, 3] = -np.inf
    out, lse = orc.lse_merge(outs, lses)
    want_lse = logsumexp(lses, axis=0)
    wts = np.exp(lses - want_lse[None])
    want = np.einsum("sr,src->rc", wts, outs)
    assert np.max(np.abs(lse - want_lse)) <= 1e-13
    assert np.max(np.abs(out - want)) <= 1e-13


# ---------------------------------------------------------------- gather
def test_page_permutation_invariance():
    w = small(41, B=2, lens=(130, 64), extra_pages=3)
    ref, ref_lse = orc.attend(w, shard=-1)
    P = w.kv.shape[0]
    perm = mi.permutation(99, 7, P)              # new position of old page p
    kv2 = np.empty_like(w.kv)
    kv2[perm] = w.kv
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    out, lse = orc.attend(w, shard=-1, kv=kv2, block_table=bt2)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_poisoned_unused_rows_are_never_read(kv_dtype):
    clean = small(42, lens=(70, 5), kv_dtype=kv_dtype, extra_pages=2)
    dirty = small(42, lens=(70, 5), kv_dtype=kv_dtype, extra_pages=2, poison=True)
    a, la = orc.attend(clean, shard=-1)
    b, lb = orc.attend(dirty, shard=-1)
    assert np.all(np.isfinite(b)) and np.array_equal(a, b) and np.array_equal(la, lb)


def test_bad_block_table_entry_is_reported():
    w = small(43, lens=(70, 5))
    w.block_table[0, 1] = w.kv.shape[0] + 5
    with pytest.raises(RuntimeError):
        orc.attend(w, shard=-1)


# ---------------------------------------------------------------- causal
def test_causal_verify_row_equals_shorter_decode():
    """Query i of a 9-token causal verify step over an L-token cache sees
    tokens t <= L - 9 + i, i.e. it equals a single-token decode of the same
    query over the first L - 8 + i tokens."""
    w = small(51, B=2, q_len=9, H=2, lens=(100, 64), causal=True)
    out, lse = orc.attend(w, shard=-1)
    for i in range(9):
        q1 = np.ascontiguousarray(w.q[:, i:i + 1])
        lens1 = (w.seq_lens - 8 + i).astype(np.int32)
        w1 = mi.Workload("q1", 2, 1, 2, lens1, 1, "interleaved", "bf16", False, 0,
                         q=q1, kv=w.kv, block_table=w.block_table)
        o1, l1 = orc.attend(w1, shard=-1)
        for b in range(2):
            for h in range(2):
                r9 = (b * 9 + i) * 2 + h
                assert np.array_equal(out[r9], o1[b * 2 + h])
                assert lse[r9] == l1[b * 2 + h]


def test_causal_mask_changes_result():
    a = small(52, B=1, q_len=3, H=2, lens=(40,), causal=True)
    b = small(52, B=1, q_len=3, H=2, lens=(40,), causal=False)
    oa, _ = orc.attend(a, shard=-1)
    ob, _ = orc.attend(b, shard=-1)
    last = slice(2 * 2, 3 * 2)                   # the last query sees everything
    assert np.array_equal(oa[last], ob[last])
    assert not np.allclose(oa[:2], ob[:2])


def test_variable_query_counts_equal_shorter_decodes_and_pad_the_rest():
    """A batch of verify steps with different draft counts, padded to one
    q_len: query i < q_lens[b] of request b sees t <= L - q_lens[b] + i, the
    same as a single-token decode of that query over the first
    L - q_lens[b] + 1 + i tokens; rows i >= q_lens[b] see nothing."""
    w = small(53, B=3, q_len=5, H=2, lens=(90, 64, 130), causal=True)
    w.q_lens = np.array([1, 5, 3], dtype=np.int32)
    out, lse = orc.attend(w, shard=-1)
    for b in range(3):
        qn = int(w.q_lens[b])
        for i in range(5):
            rows = [(b * 5 + i) * 2 + h for h in range(2)]
            if i >= qn:
                assert np.all(out[rows] == 0.0) and np.all(np.isneginf(lse[rows]))
                continue
            q1 = np.ascontiguousarray(w.q[b:b + 1, i:i + 1])
            lens1 = np.array([w.seq_lens[b] - qn + 1 + i], dtype=np.int32)
            w1 = mi.Workload("q1", 1, 1, 2, lens1, 1, "interleaved", "bf16", False, 0,
                             q=q1, kv=w.kv, block_table=np.ascontiguousarray(w.block_table[b:b + 1]))
            o1, l1 = orc.attend(w1, shard=-1)
            for h in range(2):
                assert np.array_equal(out[rows[h]], o1[h])
                assert lse[rows[h]] == l1[h]


def test_full_query_counts_equal_a_uniform_batch():
    w = small(54, B=2, q_len=4, H=2, lens=(70, 200), causal=True)
    o0, l0 = orc.attend(w, shard=-1)
    w.q_lens = np.array([4, 4], dtype=np.int32)
    o1, l1 = orc.attend(w, shard=-1)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_variable_query_counts_shard_and_merge():
    """The shard invariant holds row by row for padded batches too."""
    w = small(55, B=3, q_len=4, H=2, lens=(30, 150, 9), causal=True)
    w.q_lens = np.array([2, 4, 1], dtype=np.int32)
    ref, ref_lse = orc.attend(w, shard=-1)
    for layout in ("interleaved", "contiguous"):
        for N in (2, 3):
            parts = [orc.attend(w, shard=s, num_shards=N, layout=layout) for s in range(N)]
            o, l = orc.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
            fin = np.isfinite(ref_lse)
            assert np.array_equal(np.isneginf(l), np.isneginf(ref_lse))
            assert np.allclose(o, ref, rtol=0, atol=1e-12)
            assert np.allclose(l[fin], ref_lse[fin], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- fp8 codec
def e4m3_closed_form(c):
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_decode(codes)
    want = np.array([e4m3_closed_form(int(c)) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    torch = pytest.importorskip("torch")
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(lib), np.isnan(got))
    assert np.array_equal(lib[ok], got[ok])


def test_e4m3_encoder_round_trip_and_saturation():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = orc.e4m3_decode(codes).astype(np.float32)
    back = mi.encode_e4m3(vals)
    pos_zero = vals == 0
    assert np.array_equal(back[~pos_zero], codes[~pos_zero])
    assert mi.encode_e4m3(np.array([1000.0, -1e6, 449.0], np.float32)).tolist() == [0x7E, 0xFE, 0x7E]
    # ties round to even: 1 + 1/16 lies halfway between 1 and 1.125
    assert mi.encode_e4m3(np.array([1.0625, 1.1875], np.float32)).tolist() == [0x38, 0x3A]


def test_fp8_rows_reconstruct_within_half_ulp():
    codes, scales = mi.normal_fp8_rows(61, 2, 64, 576, 1.0)
    x = mi.normal_f32(61, 2, (64, 576), 1.0)
    recon = orc.e4m3_decode(codes).reshape(64, 576) * scales[:, None]
    assert np.allclose(scales, np.max(np.abs(x), axis=1) / 448.0, rtol=1e-6)
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals
    rel = np.abs(recon - x) / np.maximum(np.abs(x), 2.0 ** -6 * scales[:, None])
    assert np.max(rel) <= 2.0 ** -4 + 1e-6


# ------------------------------------------------------------------- W_UV
def test_wuv_projection_matches_matmul_and_commutes_with_merge():
    w = small(71, B=2, H=2, lens=(90, 33))
    w_uv = mi.normal_bf16(71, 5, (2, 512, 128), 0.02)
    wf = mi.bf16_bits_to_f32(w_uv).astype(np.float64)
    parts = [orc.attend(w, shard=s, num_shards=3, layout="interleaved") for s in range(3)]
    heads = np.tile(np.arange(2, dtype=np.int32), 2)
    merged, lse = orc.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    y = orc.project_wuv(merged, heads, w_uv)
    want = np.einsum("rc,rcj->rj", merged, wf[heads])
    assert np.max(np.abs(y - want)) <= 1e-14
    # project each shard, then merge with the same LSE weights
    projected = [orc.project_wuv(p[0], heads, w_uv) for p in parts]
    wts = np.exp(np.stack([p[1] for p in parts]) - lse[None])
    y2 = np.einsum("sr,srj->rj", wts, np.stack(projected))
    assert np.max(np.abs(y2 - y)) <= 1e-14


def test_wuv_one_hot_selects_latent_columns():
    w = small(72, B=1, H=2, lens=(40,))
    out, _ = orc.attend(w, shard=-1)
    cols = mi.permutation(72, 9, 512)[:128]
    w_uv = np.zeros((2, 512, 128), dtype=np.uint16)
    w_uv[:, cols, np.arange(128)] = 0x3F80            # bf16 1.0
    y = orc.project_wuv(out, np.array([0, 1], np.int32), w_uv)
    assert np.array_equal(y, out[:, cols])


# -------------------------------------------------------------- inputs
def test_agentic_length_mix_matches_trace_shape():
    """The stand-in length mix meets the fractions given for the agentic
    trace ("Decode Context Parallelism", section 2.1)."""
    lens = mi.agentic_lengths(2, 32)
    n = len(lens)
    assert n == 32 and lens.sum() <= 4 * 1024 * 1024
    assert abs(np.mean(lens < 65536) - 0.47) < 0.02
    assert abs(np.mean(lens < 8192) - 0.18) < 0.02
    assert 0.03 <= np.mean(lens > 262144) <= 0.04
    assert 0.05 <= np.mean(lens > 131072) <= 0.10
    assert 64 * 1024 <= np.median(lens) <= 68 * 1024
    assert lens.max() <= 1048576


def test_generator_is_deterministic_and_thread_independent():
    a = mi.normal_bf16(5, 2, (1000,), 0.5)
    b = mi.normal_bf16(5, 2, (1000,), 0.5)
    c = mi.normal_bf16(5, 2, (600,), 0.5, offset=400)
    assert np.array_equal(a, b) and np.array_equal(a[400:], c)
    x = mi.bf16_bits_to_f32(mi.normal_bf16(6, 2, (200000,), 1.0)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
