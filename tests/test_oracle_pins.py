"""Pins for the fp64 oracle: checks against what the pages and plain
mathematics fix, never against the oracle itself or the CUDA path.

Each test names the page section it follows.  A plausible slip in the oracle
(a dropped causal offset, a wrong GQA index, a transposed gather, a wrong LSE
base or merge weight) makes at least one of these fail; see
``test_oracle_mutants.py`` for that claim checked by planting such slips.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import workloads
from tests import bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# "Attention Backends", section "Code": the block-table worked example.
# ---------------------------------------------------------------------------

def _m1_inputs():
    g = _golden("m1_block_table.json")
    bs, dim, seq = g["block_size"], g["dim"], g["seq_len"]
    keys = [[math.sin(i * 3 + d) for d in range(dim)] for i in range(seq)]
    vals = [[math.cos(i * 5 + d * 2) for d in range(dim)] for i in range(seq)]
    return g, keys, vals


def _m1_pool(table, keys, vals, bs, nb, dim):
    # Unused slots hold NaN: reading one would poison the result.
    pool = np.full((nb, 2, bs, 1, dim), np.nan)
    for pos in range(len(keys)):
        blk, off = table[pos // bs], pos % bs
        pool[blk, 0, off, 0] = keys[pos]
        pool[blk, 1, off, 0] = vals[pos]
    return pool


def test_m1_slot_ranges(oracle_lib):
    g, keys, vals = _m1_inputs()
    bs, table = g["block_size"], g["block_table"]
    slots = [table[p // bs] * bs + p % bs for p in range(g["seq_len"])]
    r = g["printed_slot_ranges"]
    assert slots[0:4] == list(range(r["positions 0-3"][0], r["positions 0-3"][1] + 1))
    assert slots[4:8] == list(range(r["positions 4-7"][0], r["positions 4-7"][1] + 1))
    assert slots[8:10] == list(range(r["positions 8-9"][0], r["positions 8-9"][1] + 1))
    # The oracle's cache write puts token p at exactly that slot.
    T, d = g["seq_len"], 8
    rng = np.random.default_rng(0)
    key = rng.integers(0, 1 << 16, size=(T, 1, d), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, size=(T, 1, d), dtype=np.uint16)
    pool = np.zeros((g["num_blocks"], 2, bs, 1, d), np.uint16)
    out = oracle_lib.reshape_and_cache(key, val, pool, np.array(slots), bs)
    for p, s in enumerate(slots):
        assert np.array_equal(out[s // bs, 0, s % bs], key[p])
        assert np.array_equal(out[s // bs, 1, s % bs], val[p])
    written = {(s // bs, s % bs) for s in slots}
    for b in range(g["num_blocks"]):
        for o in range(bs):
            if (b, o) not in written:
                assert not out[b, :, o].any()


@pytest.mark.parametrize("table", [[6, 1, 4], [0, 1, 2], [7, 3, 5]])
def test_m1_paged_equals_contiguous(oracle_lib, table):
    g, keys, vals = _m1_inputs()
    bs, dim, seq, nb = g["block_size"], g["dim"], g["seq_len"], g["num_blocks"]
    scale = 1.0 / math.sqrt(dim)
    q = np.array(g["query"], np.float64).reshape(1, 1, dim)
    pool = _m1_pool(table, keys, vals, bs, nb, dim)
    out, lse = oracle_lib.paged_attention(q, pool, np.array([table]), [0, 1], [seq], scale)
    ref_o, ref_lse = bruteforce.attend(g["query"], keys, vals, scale)
    np.testing.assert_allclose(out[0, 0], ref_o, rtol=0, atol=1e-13)
    assert abs(lse[0, 0] - ref_lse) < 1e-13
    # Bit-for-bit equality with the paper's scattered table (the page's claim).
    pool0 = _m1_pool(g["block_table"], keys, vals, bs, nb, dim)
    out0, lse0 = oracle_lib.paged_attention(q, pool0, np.array([g["block_table"]]), [0, 1],
                                            [seq], scale)
    assert np.array_equal(out, out0) and np.array_equal(lse, lse0)


# ---------------------------------------------------------------------------
# "Chapter 1: attention backends", section 4.1, Fig. 5c: online softmax and
# the merge of two key blocks.
# ---------------------------------------------------------------------------

def test_fig5c_block_merge(oracle_lib):
    g = _golden("fig5c_online_softmax.json")
    v = g["values"]
    scores = [0.0, 0.0, math.log(2.0), math.log(2.0)]   # weights 1:1:2:2
    bs, nb = 2, 2
    pool = np.zeros((nb, 2, bs, 1, 1))
    for p in range(4):
        pool[p // bs, 0, p % bs, 0, 0] = scores[p]
        pool[p // bs, 1, p % bs, 0, 0] = v[p]
    q = np.ones((1, 1, 1))
    table = np.array([[0, 1]])
    part = oracle_lib.split_partials(q, pool, table, [4], 1.0, 2)
    o_a, lse_a = part[0, 0, 0, 0], part[0, 0, 0, 1]
    o_b, lse_b = part[0, 0, 1, 0], part[0, 0, 1, 1]
    assert abs(o_a - g["block_A_output"]) < 1e-12
    assert abs(lse_a - math.log(2.0)) < 1e-12
    assert abs(o_b - 35.0) < 1e-12 and abs(lse_b - math.log(4.0)) < 1e-12
    out, lse = oracle_lib.lse_merge(part)
    assert abs(out[0, 0, 0] - 170.0 / 6.0) < 1e-12
    assert abs(out[0, 0, 0] - g["merged_output_approx"]) < 5e-3
    assert abs(lse[0, 0] - math.log(6.0)) < 1e-12
    assert abs(math.exp(lse_a - lse[0, 0]) - g["share_of_A_after_B"]) < 1e-12
    # The merged result equals attention over the whole row (Fig. 5a).
    full_o, full_lse = oracle_lib.paged_attention(q, pool, table, [0, 1], [4], 1.0)
    assert abs(full_o[0, 0, 0] - out[0, 0, 0]) < 1e-12
    assert abs(full_lse[0, 0] - lse[0, 0]) < 1e-12


# ---------------------------------------------------------------------------
# Closed forms of O = softmax(Q K^T / sqrt(d) + M) V ("Chapter 1", 2.1).
# ---------------------------------------------------------------------------

def _f64(bits):
    return workloads.bf16_bits_to_f32(bits).astype(np.float64)


def _gather(pool, table_row, seq, bs):
    """numpy fancy-index gather of one request's K, V: [seq, Hkv, d]."""
    pos = np.arange(seq)
    blk = np.asarray(table_row)[pos // bs]
    return pool[blk, 0, pos % bs], pool[blk, 1, pos % bs]


def test_zero_query_gives_mean_of_visible_rows_causal(oracle_lib):
    # q = 0: every visible score is 0, so o is the mean of the visible V rows
    # and lse = ln(#visible).  With bottom-right causal alignment row j of a
    # request with context c sees c + j + 1 positions.
    b = workloads.make_paged_batch("zq", 11, [5, 40, 33], [5, 7, 1], 4, 2, 16, 16)
    q = np.zeros_like(b.q)
    out, lse = oracle_lib.paged_attention(q, b.pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    pool = _f64(b.pool)
    grp = b.num_q_heads // b.num_kv_heads
    for i in range(b.num_seqs):
        _, V = _gather(pool, b.block_table[i], b.seq_lens[i], b.block_size)
        ctx = b.seq_lens[i] - b.query_lens[i]
        for j in range(b.query_lens[i]):
            row = b.query_start_loc[i] + j
            n = ctx + j + 1
            for h in range(b.num_q_heads):
                np.testing.assert_allclose(out[row, h], V[:n, h // grp].mean(axis=0),
                                           rtol=0, atol=1e-13)
                assert abs(lse[row, h] - math.log(n)) < 1e-13
    # Non-causal: every row sees all seq_len positions.
    out, lse = oracle_lib.paged_attention(q, b.pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, causal=False)
    for i in range(b.num_seqs):
        rows = range(b.query_start_loc[i], b.query_start_loc[i + 1])
        for row in rows:
            assert np.allclose(lse[row], math.log(b.seq_lens[i]), atol=1e-13)


def test_single_token_returns_that_value_row(oracle_lib):
    b = workloads.make_paged_batch("one", 12, [1, 1], [1, 1], 4, 2, 64, 16, num_blocks=5)
    out, lse = oracle_lib.paged_attention(b.q, b.pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    pool, q = _f64(b.pool), _f64(b.q)
    for i in range(2):
        blk = b.block_table[i, 0]
        for h in range(4):
            k, v = pool[blk, 0, 0, h // 2], pool[blk, 1, 0, h // 2]
            assert np.array_equal(out[i, h], v)            # weight exactly 1
            assert abs(lse[i, h] - b.scale * float(np.dot(q[i, h], k))) < 1e-12


def test_gqa_head_mapping_and_row_sums(oracle_lib):
    # V constant per kv head (value g + 1): q head h must return (h // grp) + 1.
    # V = 1 everywhere checks that the softmax weights sum to one.
    b = workloads.make_paged_batch("gqa", 13, [37, 64], [3, 2], 8, 2, 16, 16)
    pool = _f64(b.pool)
    for g in range(b.num_kv_heads):
        pool[:, 1, :, g, :] = g + 1.0
    q = _f64(b.q)
    out, _ = oracle_lib.paged_attention(q, pool, b.block_table, b.query_start_loc,
                                        b.seq_lens, b.scale)
    for h in range(8):
        np.testing.assert_allclose(out[:, h], h // 4 + 1.0, rtol=0, atol=1e-13)


def test_gqa_equals_replicated_mha(oracle_lib):
    b = workloads.make_paged_batch("rep", 14, [29, 50], [4, 1], 6, 2, 32, 16)
    pool = b.pool
    rep = np.repeat(pool, 3, axis=3)       # kv head g copied to heads 3g..3g+2
    o1, l1 = oracle_lib.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                        b.seq_lens, b.scale)
    o2, l2 = oracle_lib.paged_attention(b.q, rep, b.block_table, b.query_start_loc,
                                        b.seq_lens, b.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_matches_torch_sdpa_on_tiny_workload(oracle_lib):
    # Library routine: torch's scaled_dot_product_attention in fp64 over the
    # contiguous K/V with an explicit bottom-right causal mask.
    b = workloads.tiny_paged()
    pool = oracle_lib.reshape_and_cache(b.key, b.value, b.pool,
                                        b.slot_mapping, b.block_size)
    out, lse = oracle_lib.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    P, q = _f64(pool), _f64(b.q)
    grp = b.num_q_heads // b.num_kv_heads
    for i in range(b.num_seqs):
        K, V = _gather(P, b.block_table[i], b.seq_lens[i], b.block_size)
        rows = slice(b.query_start_loc[i], b.query_start_loc[i + 1])
        qi = torch.from_numpy(q[rows]).permute(1, 0, 2)                 # [Hq, L, d]
        Ki = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(grp, 0)
        Vi = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(grp, 0)
        L, S = qi.shape[1], Ki.shape[1]
        mask = torch.arange(S)[None, :] <= (S - L + torch.arange(L))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qi, Ki, Vi, attn_mask=mask, scale=b.scale)
        np.testing.assert_allclose(out[rows], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        s = torch.einsum("hld,hsd->hls", qi, Ki) * b.scale
        s = s.masked_fill(~mask, -math.inf)
        np.testing.assert_allclose(lse[rows], torch.logsumexp(s, -1).T.numpy(), rtol=0,
                                   atol=1e-12)


def test_matches_pure_python_bruteforce_on_tiny_workload(oracle_lib):
    b = workloads.tiny_paged()
    pool = oracle_lib.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    out, lse = oracle_lib.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    P, q = _f64(pool), _f64(b.q)
    grp = b.num_q_heads // b.num_kv_heads
    for i in range(b.num_seqs):
        seq, qlen = int(b.seq_lens[i]), int(b.query_lens[i])
        for j in range(qlen):
            row = int(b.query_start_loc[i]) + j
            n = seq - qlen + j + 1
            for h in range(b.num_q_heads):
                keys, vals = [], []
                for p in range(n):
                    blk = int(b.block_table[i][p // b.block_size])
                    keys.append(list(P[blk, 0, p % b.block_size, h // grp]))
                    vals.append(list(P[blk, 1, p % b.block_size, h // grp]))
                o, l = bruteforce.attend(list(q[row, h]), keys, vals, b.scale)
                np.testing.assert_allclose(out[row, h], o, rtol=0, atol=1e-12)
                assert abs(lse[row, h] - l) < 1e-12


def test_block_permutation_invariance(oracle_lib):
    b = workloads.make_paged_batch("perm", 15, [70, 33, 16], [3, 33, 1], 4, 4, 16, 16,
                                   num_blocks=12)
    o1, l1 = oracle_lib.paged_attention(b.q, b.pool, b.block_table, b.query_start_loc,
                                        b.seq_lens, b.scale)
    perm = np.random.default_rng(3).permutation(b.num_blocks)
    new_pool = np.empty_like(b.pool)
    new_pool[perm] = b.pool                     # block k moves to perm[k]
    table = np.where(b.block_table >= 0, perm[np.maximum(b.block_table, 0)], -1)
    o2, l2 = oracle_lib.paged_attention(b.q, new_pool, table, b.query_start_loc,
                                        b.seq_lens, b.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---------------------------------------------------------------------------
# Split-KV ("Chapter 1", 3.1; "Triton and MLA", data flow): splitting adds
# parallelism but every key still takes part, so split + LSE merge equals the
# unsplit result, and one split is the unsplit result.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 7, 256])
def test_split_then_merge_equals_unsplit(oracle_lib, S):
    b = workloads.make_paged_batch("split", 16, [300, 17, 1, 64], [1, 1, 1, 1], 8, 2, 32, 16)
    unsplit_o, unsplit_l = oracle_lib.paged_attention(b.q, b.pool, b.block_table,
                                                      b.query_start_loc, b.seq_lens, b.scale)
    part = oracle_lib.split_partials(b.q, b.pool, b.block_table, b.seq_lens, b.scale, S)
    o, l = oracle_lib.lse_merge(part)
    np.testing.assert_allclose(o, unsplit_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, unsplit_l, rtol=0, atol=1e-12)
    if S == 1:
        assert np.array_equal(part[:, :, 0, :-1], unsplit_o)
        assert np.array_equal(part[:, :, 0, -1], unsplit_l)
    # Split boundaries: one chunk C = bs * ceil(ceil(max_seq / S) / bs) for
    # the whole batch; splits past a request's end are empty (o = 0,
    # lse = -inf).
    per = -(-int(b.seq_lens.max()) // S)
    chunk = -(-per // b.block_size) * b.block_size
    P, q = _f64(b.pool), _f64(b.q)
    grp = b.num_q_heads // b.num_kv_heads
    for i, seq in enumerate(b.seq_lens):
        K, _ = _gather(P, b.block_table[i], seq, b.block_size)
        for s in range(S):
            a = min(s * chunk, seq)
            e = seq if s == S - 1 else min((s + 1) * chunk, seq)
            empty = a >= e
            assert np.isneginf(part[i, :, s, -1]).all() == empty
            if empty:
                assert not part[i, :, s, :-1].any()
                continue
            # The split's LSE is the log-sum-exp of exactly its tokens' scores.
            for h in range(b.num_q_heads):
                sc = b.scale * K[a:e, h // grp] @ q[i, h]
                ref = sc.max() + math.log(np.exp(sc - sc.max()).sum())
                assert abs(part[i, h, s, -1] - ref) < 1e-12
    # An understated max_seq_len only makes the last split longer.
    part2 = oracle_lib.split_partials(b.q, b.pool, b.block_table, b.seq_lens, b.scale, S,
                                      max_seq_len=17)
    o2, l2 = oracle_lib.lse_merge(part2)
    np.testing.assert_allclose(o2, unsplit_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, unsplit_l, rtol=0, atol=1e-12)


def test_merge_ignores_empty_and_handles_all_empty(oracle_lib):
    part = np.zeros((2, 1, 3, 3))
    part[0, 0, 0] = [1.0, 2.0, 0.5]
    part[0, 0, 1] = [0.0, 0.0, -np.inf]
    part[0, 0, 2] = [3.0, 4.0, 0.5]
    part[1, 0, :, 2] = -np.inf
    o, l = oracle_lib.lse_merge(part)
    np.testing.assert_allclose(o[0, 0], [2.0, 3.0], atol=1e-15)
    assert abs(l[0, 0] - (0.5 + math.log(2.0))) < 1e-15
    assert not o[1].any() and np.isneginf(l[1, 0])


# ---------------------------------------------------------------------------
# MLA ("Triton and MLA", data flow): MQA over one [kv_c | k_pe] vector, value
# = its first kv_lora_rank entries.
# ---------------------------------------------------------------------------

def test_mla_equals_generic_single_kv_head(oracle_lib):
    b = workloads.make_mla_batch("mla", 17, [70, 5, 128], 4, kv_lora_rank=40, rope_dim=8,
                                 block_size=16)
    o, l = oracle_lib.mla_decode(b.q, b.pool, b.block_table, b.seq_lens, b.scale, 40, 8)
    # Standard layout with one kv head, K = V = the whole 48-wide row.
    std = np.stack([b.pool, b.pool], axis=1)[:, :, :, None, :]
    qsl = np.arange(b.batch + 1)
    go, gl = oracle_lib.paged_attention(b.q, std, b.block_table, qsl, b.seq_lens, b.scale)
    assert np.array_equal(o, go[:, :, :40]) and np.array_equal(l, gl)


def test_mla_matches_bruteforce(oracle_lib):
    b = workloads.make_mla_batch("mla_bf", 18, [9, 33], 3, kv_lora_rank=16, rope_dim=8,
                                 block_size=16)
    o, l = oracle_lib.mla_decode(b.q, b.pool, b.block_table, b.seq_lens, b.scale, 16, 8)
    P, q = _f64(b.pool), _f64(b.q)
    for i in range(b.batch):
        rows = [P[b.block_table[i][p // 16], p % 16] for p in range(b.seq_lens[i])]
        for h in range(3):
            ro, rl = bruteforce.attend(list(q[i, h]), [list(r) for r in rows],
                                       [list(r[:16]) for r in rows], b.scale)
            np.testing.assert_allclose(o[i, h], ro, rtol=0, atol=1e-12)
            assert abs(l[i, h] - rl) < 1e-12


# ---------------------------------------------------------------------------
# Cache write ("Attention Backends", paged-kernel contract step 1).
# ---------------------------------------------------------------------------

def test_cache_write_matches_numpy_scatter(oracle_lib):
    b = workloads.tiny_paged()
    out = oracle_lib.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    ref = b.pool.copy()
    s = b.slot_mapping
    ref[s // b.block_size, 0, s % b.block_size] = b.key
    ref[s // b.block_size, 1, s % b.block_size] = b.value
    assert np.array_equal(out, ref)
    skip = b.slot_mapping.copy()
    skip[1] = -1
    out2 = oracle_lib.reshape_and_cache(b.key, b.value, b.pool, skip, b.block_size)
    blk, off = s[1] // b.block_size, s[1] % b.block_size
    assert np.array_equal(out2[blk, :, off], b.pool[blk, :, off])
    bad = b.slot_mapping.copy()
    bad[0] = b.num_blocks * b.block_size
    with pytest.raises(ValueError):
        oracle_lib.reshape_and_cache(b.key, b.value, b.pool, bad, b.block_size)


def test_empty_request_gives_neg_inf_lse(oracle_lib):
    b = workloads.make_paged_batch("empty", 19, [0, 20], [0, 1], 2, 1, 16, 16, num_blocks=3)
    part = oracle_lib.split_partials(np.zeros((2, 2, 16), np.uint16), b.pool, b.block_table,
                                     b.seq_lens, b.scale, 3)
    o, l = oracle_lib.lse_merge(part)
    assert np.isneginf(l[0]).all() and not o[0].any()
    assert np.isfinite(l[1]).all()


# ---------------------------------------------------------------------------
# fp8 (e4m3) cache: "Triton and MLA", data flow -- the decode kernel always
# gets the layer's k_scale / v_scale and dequantises an fp8 cache itself.
# The e4m3 format and its rounding are pinned against torch's float8_e4m3fn
# (a library implementation of the OCP FP8 format), never against the oracle.
# ---------------------------------------------------------------------------

def _torch_e4m3_codes(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def test_fp8_decode_all_codes_match_torch(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    mine, ref = oracle_lib.e4m3_decode(codes), _torch_e4m3_values(codes)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9   # largest, smallest


def test_fp8_encode_matches_torch_and_ties_to_even(oracle_lib):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-14, 6, 100000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    assert np.array_equal(oracle_lib.e4m3_encode(x), _torch_e4m3_codes(x))
    # Every finite value, and every midpoint between neighbours (a tie, which
    # must go to the even code), with both signs.
    vals = _torch_e4m3_values(np.arange(0x7F, dtype=np.uint8))   # 0 .. 448
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    pts = np.concatenate([vals.astype(np.float32), mids])
    pts = np.concatenate([pts, -pts])
    assert np.array_equal(oracle_lib.e4m3_encode(pts), _torch_e4m3_codes(pts))
    assert oracle_lib.e4m3_encode(np.array([1.0625], np.float32))[0] == 0x38   # 1.0625 -> 1.0


def test_fp8_encode_saturates_and_keeps_signed_zero(oracle_lib):
    x = np.array([448.0, 460.0, 479.0, 1e6, 3e38, -449.0, -1e30, 0.0, -0.0, 1e-30, -1e-30],
                 np.float32)
    assert list(oracle_lib.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE,
                                                0x00, 0x80, 0x00, 0x80]


def test_fp8_cache_write_matches_torch_quantisation(oracle_lib):
    b = workloads.tiny_paged()
    ks, vs = 0.37, 0.61
    pool0 = np.full(b.pool.shape, 0x5A, np.uint8)
    out = oracle_lib.reshape_and_cache_fp8(b.key, b.value, pool0, b.slot_mapping, b.block_size,
                                           ks, vs)
    key32 = workloads.bf16_bits_to_f32(b.key)
    val32 = workloads.bf16_bits_to_f32(b.value)
    ref = pool0.copy()
    s = b.slot_mapping
    ref[s // b.block_size, 0, s % b.block_size] = _torch_e4m3_codes(key32 / np.float32(ks))
    ref[s // b.block_size, 1, s % b.block_size] = _torch_e4m3_codes(val32 / np.float32(vs))
    assert np.array_equal(out, ref)
    skip = s.copy()
    skip[0] = -1
    out2 = oracle_lib.reshape_and_cache_fp8(b.key, b.value, pool0, skip, b.block_size, ks, vs)
    assert np.array_equal(out2[s[0] // b.block_size, :, s[0] % b.block_size],
                          pool0[s[0] // b.block_size, :, s[0] % b.block_size])


def _fp8_decode_batch():
    b = workloads.make_paged_batch("fp8", 23, [1, 17, 40, 64], [1, 1, 1, 1], 4, 2, 64, 16,
                                   num_blocks=12)
    rng = np.random.default_rng(5)
    pool = rng.integers(0, 256, size=b.pool.shape, dtype=np.uint8)
    pool[(pool & 0x7F) == 0x7F] = 0x3C        # no NaN codes
    return b, pool


def test_fp8_split_partials_equal_bf16_path_for_power_of_two_scales(oracle_lib):
    # With scales 2^k every dequantised entry is exactly a bf16 value, so the
    # fp8 path must agree exactly with the bf16 path on that bf16 pool.
    b, pool = _fp8_decode_batch()
    ks, vs = 0.125, 2.0
    vals = _torch_e4m3_values(pool)
    vals[:, 0] *= ks
    vals[:, 1] *= vs
    bits = workloads.f32_to_bf16_bits(vals.astype(np.float32))
    assert np.array_equal(workloads.bf16_bits_to_f32(bits).astype(np.float64), vals)
    q = b.q.reshape(b.num_seqs, b.num_q_heads, b.head_size)
    p8 = oracle_lib.split_partials_fp8(q, pool, b.block_table, b.seq_lens, b.scale, ks, vs, 3)
    p16 = oracle_lib.split_partials(q, bits, b.block_table, b.seq_lens, b.scale, 3)
    assert np.array_equal(p8, p16)


def test_fp8_decode_matches_torch_sdpa(oracle_lib):
    b, pool = _fp8_decode_batch()
    ks, vs = float(np.float32(0.37)), float(np.float32(0.61))   # scales are fp32 values
    q = b.q.reshape(b.num_seqs, b.num_q_heads, b.head_size)
    o, lse = oracle_lib.lse_merge(
        oracle_lib.split_partials_fp8(q, pool, b.block_table, b.seq_lens, b.scale, ks, vs, 2))
    vals = _torch_e4m3_values(pool)
    g = b.num_q_heads // b.num_kv_heads
    for i in range(b.num_seqs):
        n = int(b.seq_lens[i])
        pos = np.arange(n)
        blk, off = b.block_table[i, pos // b.block_size], pos % b.block_size
        K = torch.from_numpy(vals[blk, 0, off] * ks)          # [n, Hkv, d]
        V = torch.from_numpy(vals[blk, 1, off] * vs)
        qi = torch.from_numpy(workloads.bf16_bits_to_f32(q[i]).astype(np.float64))   # [Hq, d]
        for h in range(b.num_q_heads):
            s = (K[:, h // g] @ qi[h]) * b.scale
            ref_o = torch.softmax(s, 0) @ V[:, h // g]
            assert np.allclose(o[i, h], ref_o.numpy(), rtol=0, atol=1e-12)
            assert abs(lse[i, h] - torch.logsumexp(s, 0).item()) < 1e-12


# ---------------------------------------------------------------- sliding window
# Reading: a row at position p sees p - W < p' <= p (the W newest positions
# a causal row sees); the pages name the parameter only.

def _window_batch():
    # Ragged lengths around the window sizes used below, queries inside and at
    # the end of each request.
    return workloads.make_paged_batch("window_pins", 61, [1, 9, 23, 40], [1, 5, 23, 7], 4, 2,
                                      16, 8, num_blocks=24, scale=0.3)


def test_window_matches_torch_sdpa_with_banded_mask(oracle_lib):
    b = _window_batch()
    pool = oracle_lib.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    P, q = _f64(pool), _f64(b.q)
    grp = b.num_q_heads // b.num_kv_heads
    for W in (1, 3, 8, 17):
        out, lse = oracle_lib.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                              b.seq_lens, b.scale, window=W)
        for i in range(b.num_seqs):
            K, V = _gather(P, b.block_table[i], b.seq_lens[i], b.block_size)
            rows = slice(b.query_start_loc[i], b.query_start_loc[i + 1])
            qi = torch.from_numpy(q[rows]).permute(1, 0, 2)
            Ki = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(grp, 0)
            Vi = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(grp, 0)
            L, S = qi.shape[1], Ki.shape[1]
            pos = (S - L + torch.arange(L))[:, None]
            key = torch.arange(S)[None, :]
            mask = (key <= pos) & (key > pos - W)
            ref = torch.nn.functional.scaled_dot_product_attention(
                qi, Ki, Vi, attn_mask=mask, scale=b.scale)
            np.testing.assert_allclose(out[rows], ref.permute(1, 0, 2).numpy(), rtol=0,
                                       atol=1e-12)
            s = torch.einsum("hld,hsd->hls", qi, Ki) * b.scale
            s = s.masked_fill(~mask, -math.inf)
            np.testing.assert_allclose(lse[rows], torch.logsumexp(s, -1).T.numpy(), rtol=0,
                                       atol=1e-12)


def test_window_brute_force(oracle_lib):
    b = _window_batch()
    pool = oracle_lib.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    P, q = _f64(pool), _f64(b.q)
    grp = b.num_q_heads // b.num_kv_heads
    W = 5
    out, lse = oracle_lib.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, window=W)
    for i in range(b.num_seqs):
        K, V = _gather(P, b.block_table[i], b.seq_lens[i], b.block_size)
        q0, q1 = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
        for j in range(q0, q1):
            p = int(b.seq_lens[i]) - (q1 - q0) + (j - q0)
            lo = max(0, p - W + 1)
            for h in range(b.num_q_heads):
                keys = [list(K[t, h // grp]) for t in range(lo, p + 1)]
                vals = [list(V[t, h // grp]) for t in range(lo, p + 1)]
                o, l = bruteforce.attend(list(q[j, h]), keys, vals, b.scale)
                np.testing.assert_allclose(out[j, h], o, rtol=0, atol=1e-12)
                assert abs(lse[j, h] - l) < 1e-12


def test_window_closed_forms(oracle_lib):
    b = _window_batch()
    pool = oracle_lib.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    args = (b.block_table, b.query_start_loc, b.seq_lens, b.scale)
    full = oracle_lib.paged_attention(b.q, pool, *args)
    # A window at least as long as every sequence changes nothing (bit-exact).
    wide = oracle_lib.paged_attention(b.q, pool, *args, window=int(b.seq_lens.max()))
    assert np.array_equal(full[0], wide[0]) and np.array_equal(full[1], wide[1])
    # W = 1: each row returns its own V row exactly, lse = scale q.k.
    P, q = _f64(pool), _f64(b.q)
    grp = b.num_q_heads // b.num_kv_heads
    one = oracle_lib.paged_attention(b.q, pool, *args, window=1)
    # q = 0: the mean of the window's V rows, lse = ln(#positions in the window).
    zq = np.zeros_like(b.q)
    W = 6
    zero = oracle_lib.paged_attention(zq, pool, *args, window=W)
    for i in range(b.num_seqs):
        K, V = _gather(P, b.block_table[i], b.seq_lens[i], b.block_size)
        q0, q1 = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
        for j in range(q0, q1):
            p = int(b.seq_lens[i]) - (q1 - q0) + (j - q0)
            lo = max(0, p - W + 1)
            for h in range(b.num_q_heads):
                assert np.array_equal(one[0][j, h], V[p, h // grp])
                assert abs(one[1][j, h] - b.scale * math.fsum(q[j, h] * K[p, h // grp])) < 1e-12
                np.testing.assert_allclose(zero[0][j, h], V[lo:p + 1, h // grp].mean(0), rtol=0,
                                           atol=1e-14)
                assert abs(zero[1][j, h] - math.log(p + 1 - lo)) < 1e-14


def test_window_is_causal_only(oracle_lib):
    b = _window_batch()
    with pytest.raises(ValueError):
        oracle_lib.paged_attention(b.q, b.pool, b.block_table, b.query_start_loc, b.seq_lens,
                                   b.scale, causal=False, window=4)


# ---------------------------------------------------------------- MLA cache write

def test_mla_cache_write_matches_numpy_scatter(oracle_lib):
    m = workloads.make_mla_batch("mla_w", 71, [1, 64, 65, 130], 4, block_size=64)
    kv_c, k_pe, slots = workloads.mla_new_tokens(m)
    out = oracle_lib.mla_cache_write(kv_c, k_pe, m.pool, slots, m.block_size)
    ref = m.pool.copy()
    ref[slots // 64, slots % 64, :512] = kv_c
    ref[slots // 64, slots % 64, 512:] = k_pe
    assert np.array_equal(out, ref)
    skip = slots.copy()
    skip[2] = -1
    out2 = oracle_lib.mla_cache_write(kv_c, k_pe, m.pool, skip, m.block_size)
    assert np.array_equal(out2[slots[2] // 64, slots[2] % 64], m.pool[slots[2] // 64,
                                                                      slots[2] % 64])
    bad = slots.copy()
    bad[0] = m.num_blocks * 64
    with pytest.raises(ValueError):
        oracle_lib.mla_cache_write(kv_c, k_pe, m.pool, bad, m.block_size)


def test_mla_cache_write_then_decode_of_one_token(oracle_lib):
    # A request of length 1 whose only token is the one just written: the MLA
    # output is that token's kv_c exactly (the value is the first 512 entries
    # of the row) and the LSE is scale * q . [kv_c | k_pe].
    m = workloads.make_mla_batch("mla_w1", 72, [1, 1, 40], 2, block_size=64)
    kv_c, k_pe, slots = workloads.mla_new_tokens(m)
    pool = oracle_lib.mla_cache_write(kv_c, k_pe, m.pool, slots, m.block_size)
    o, l = oracle_lib.mla_decode(m.q, pool, m.block_table, m.seq_lens, m.scale)
    row = np.concatenate([_f64(kv_c), _f64(k_pe)], axis=1)
    q = _f64(m.q)
    for i in (0, 1):
        for h in range(2):
            assert np.array_equal(o[i, h], row[i, :512])
            assert abs(l[i, h] - m.scale * math.fsum(q[i, h] * row[i])) < 1e-12


# ---------------------------------------------------------------- MLA prefill
# Multi-head formulation: each head's key is [w_kv_b[h, :dn] c | k_pe], its
# value w_kv_b[h, dn:] c, the expanded parts rounded to bf16 (the dtype of the
# projection's output).

def _mla_prefill_tiny(oracle_lib):
    """A ragged prefill batch (causal rows inside and at the end of each
    request) with its new latent rows already written."""
    b = workloads.make_mla_prefill_batch("mla_pf", 81, [20, 9, 37], [5, 9, 1], 3,
                                         kv_lora_rank=16, rope_dim=8, qk_nope_dim=8, v_dim=6,
                                         block_size=16)
    pool = oracle_lib.mla_cache_write(b.kv_c, b.k_pe, b.pool, b.slot_mapping, b.block_size)
    return b, pool


def _py_round_bf16(x):
    """Nearest bf16 value of a float (8 significant bits, ties to even),
    written independently of the oracle's."""
    if x == 0.0:
        return x
    m, e = math.frexp(x)                 # x = m * 2^e, 0.5 <= |m| < 1
    scaled = m * 256.0                   # 8 significant bits above the point
    r = round(scaled)                    # Python rounds halves to even
    return math.ldexp(r, e - 8)


def test_round_bf16_matches_torch_on_float32_values(oracle_lib):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3.0 + 2.0 ** -7],
                    np.float32)
    x = np.concatenate([x, ties]).astype(np.float64)
    mine = oracle_lib.round_bf16(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(mine, ref)
    assert all(_py_round_bf16(v) == r for v, r in zip(x[-4:], mine[-4:]))


def test_mla_prefill_matches_bruteforce(oracle_lib):
    b, pool = _mla_prefill_tiny(oracle_lib)
    out, lse = oracle_lib.mla_prefill(b.q, pool, b.w_kv_b, b.block_table, b.query_start_loc,
                                      b.seq_lens, b.scale)
    P, q, W = _f64(pool), _f64(b.q), _f64(b.w_kv_b)
    R, dn = b.kv_lora_rank, b.qk_nope_dim
    for i in range(b.num_seqs):
        n = int(b.seq_lens[i])
        rows = [P[b.block_table[i][p // 16], p % 16] for p in range(n)]
        q0, q1 = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
        for h in range(b.num_heads):
            keys, vals = [], []
            for r in rows:
                c = list(r[:R])
                kn = [_py_round_bf16(math.fsum(W[h, e, k] * c[k] for k in range(R)))
                      for e in range(dn)]
                v = [_py_round_bf16(math.fsum(W[h, dn + e, k] * c[k] for k in range(R)))
                     for e in range(b.v_dim)]
                keys.append(kn + list(r[R:]))
                vals.append(v)
            for j in range(q0, q1):
                vis = n - (q1 - q0) + (j - q0) + 1
                o, l = bruteforce.attend(list(q[j, h]), keys[:vis], vals[:vis], b.scale)
                np.testing.assert_allclose(out[j, h], o, rtol=0, atol=1e-12)
                assert abs(lse[j, h] - l) < 1e-12


def test_mla_prefill_equals_absorbed_formulation(oracle_lib):
    # "The same mathematics" in the decode formulation: q_abs = [W_UK^T q_nope
    # | q_pe] against the latent rows themselves (one shared kv head, key =
    # whole row, value = its first R entries), then o = W_UV o_latent.  Exact
    # (unrounded) expansion on the prefill side.
    b, pool = _mla_prefill_tiny(oracle_lib)
    out, lse = oracle_lib.mla_prefill(b.q, pool, b.w_kv_b, b.block_table, b.query_start_loc,
                                      b.seq_lens, b.scale, round_kv=False)
    P, q, W = _f64(pool), _f64(b.q), _f64(b.w_kv_b)
    R, dn, dr = b.kv_lora_rank, b.qk_nope_dim, b.rope_dim
    q_abs = np.concatenate([np.einsum("her,the->thr", W[:, :dn], q[:, :, :dn]), q[:, :, dn:]],
                           axis=2)                                   # [T, H, R + dr]
    std = np.stack([P, P], axis=1)[:, :, :, None, :]                 # [nb, 2, bs, 1, R + dr]
    o_lat, l_abs = oracle_lib.paged_attention(q_abs, std, b.block_table, b.query_start_loc,
                                              b.seq_lens, b.scale)
    o_abs = np.einsum("hvr,thr->thv", W[:, dn:], o_lat[:, :, :R])
    np.testing.assert_allclose(out, o_abs, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, l_abs, rtol=0, atol=1e-12)


def test_mla_prefill_matches_torch_sdpa(oracle_lib):
    b, pool = _mla_prefill_tiny(oracle_lib)
    out, lse = oracle_lib.mla_prefill(b.q, pool, b.w_kv_b, b.block_table, b.query_start_loc,
                                      b.seq_lens, b.scale, round_kv=False)
    P, q, W = _f64(pool), _f64(b.q), _f64(b.w_kv_b)
    R, dn = b.kv_lora_rank, b.qk_nope_dim
    for i in range(b.num_seqs):
        n = int(b.seq_lens[i])
        pos = np.arange(n)
        rows = torch.from_numpy(P[b.block_table[i, pos // 16], pos % 16])        # [n, R + dr]
        Wt = torch.from_numpy(W)
        K = torch.cat([torch.einsum("her,nr->hne", Wt[:, :dn], rows[:, :R]),
                       rows[None, :, R:].expand(b.num_heads, n, -1)], -1)     # [H, n, dk]
        V = torch.einsum("hvr,nr->hnv", Wt[:, dn:], rows[:, :R])               # [H, n, dv]
        q0, q1 = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
        qi = torch.from_numpy(q[q0:q1]).permute(1, 0, 2)                       # [H, L, dk]
        L = q1 - q0
        mask = torch.arange(n)[None, :] <= (n - L + torch.arange(L))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qi, K, V, attn_mask=mask,
                                                               scale=b.scale)
        np.testing.assert_allclose(out[q0:q1], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        s = torch.einsum("hld,hnd->hln", qi, K) * b.scale
        s = s.masked_fill(~mask, -math.inf)
        np.testing.assert_allclose(lse[q0:q1], torch.logsumexp(s, -1).T.numpy(), rtol=0,
                                   atol=1e-12)
