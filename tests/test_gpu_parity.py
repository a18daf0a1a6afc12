"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs.  Cache writes must be bit-exact; attention outputs
must meet the tolerances in ``tests/parity.py``.

Unused pool blocks and the unused tail of every request's last block are
filled with NaN, so a kernel that read anything outside a request's first
seq_len tokens would produce NaN and fail.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import (BF16_NAN, assert_lse_close, assert_out_close, bf16_bits, bf16_to_f64,
                          to_dev, to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_50_gb300 import build
    build.build()
    import paged_kv_cache_50_gb300 as pa
    pa.lib()
    assert pa.pa_get_device_error() == 0
    return pa


def _poison(b):
    pool = b.pool.copy()
    used = np.zeros((b.num_blocks, b.block_size), bool)
    for i in range(b.num_seqs):
        n = int(b.seq_lens[i])
        if n == 0:
            continue
        pos = np.arange(n)
        used[b.block_table[i, pos // b.block_size], pos % b.block_size] = True
    nb, two, bs, hkv, d = pool.shape
    pv = pool.transpose(0, 2, 1, 3, 4)          # [nb, bs, 2, Hkv, d] view
    pv[~used] = BF16_NAN
    return pool


class Dev:
    """A standard-layout batch on the device, after the step's cache write."""

    def __init__(self, pa, b, poison=True):
        self.b = b
        pool = _poison(b) if poison else b.pool.copy()
        self.host_pool_before = pool
        self.pool = to_dev_bf16(pool)
        self.q = to_dev_bf16(b.q)
        self.key = to_dev_bf16(b.key)
        self.value = to_dev_bf16(b.value)
        self.slots = to_dev(b.slot_mapping, torch.int64)
        self.table = to_dev(b.block_table, torch.int32)
        self.qsl = to_dev(b.query_start_loc, torch.int32)
        self.seq = to_dev(b.seq_lens, torch.int32)
        pa.pa_reshape_and_cache(self.key, self.value, self.pool, self.slots)

    def ref_pool(self):
        b = self.b
        return oracle.reshape_and_cache(b.key, b.value, self.host_pool_before, b.slot_mapping,
                                        b.block_size)


# ---------------------------------------------------------------------------
# Cache write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("make", [workloads.tiny_paged, workloads.gqa_decode,
                                  workloads.chunked_prefill],
                         ids=["tiny", "gqa_decode", "chunked_prefill"])
def test_cache_write_bit_exact(pa, make):
    b = make()
    d = Dev(pa, b)
    got = bf16_bits(d.pool)
    ref = d.ref_pool()
    assert np.array_equal(got, ref)
    assert pa.pa_get_device_error() == 0


def test_cache_write_skip_and_out_of_range(pa):
    b = workloads.tiny_paged()
    slots = b.slot_mapping.copy()
    slots[2] = -1                                   # skipped
    slots[4] = b.num_blocks * b.block_size + 3      # outside the pool: flagged, not written
    pool = b.pool.copy()
    d_pool = to_dev_bf16(pool)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key), to_dev_bf16(b.value), d_pool,
                            to_dev(slots, torch.int64))
    assert pa.pa_get_device_error() == pa.PA_DEVERR_SLOT
    keep = slots.copy()
    keep[4] = -1
    ref = oracle.reshape_and_cache(b.key, b.value, pool, keep, b.block_size)
    assert np.array_equal(bf16_bits(d_pool), ref)
    assert pa.pa_get_device_error() == 0             # read-and-clear


# ---------------------------------------------------------------------------
# Varlen paged attention
# ---------------------------------------------------------------------------

def _varlen(pa, d, causal=True):
    b = d.b
    out, lse = pa.pa_varlen_fwd(d.q, d.pool, d.table, d.qsl, d.seq, int(b.query_lens.max()),
                                b.scale, causal=causal)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_tiny_workload(pa, causal):
    b = workloads.tiny_paged()
    d = Dev(pa, b)
    out, lse = _varlen(pa, d, causal)
    ref_o, ref_l = oracle.paged_attention(b.q, d.ref_pool(), b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, causal=causal)
    assert_out_close(out, ref_o, "tiny out")
    assert_lse_close(lse, ref_l, "tiny lse")
    assert pa.pa_get_device_error() == 0


VARLEN_CASES = {
    # name: (seed, seq_lens, query_lens, Hq, Hkv, d, bs)
    "ragged_d128_g4": (21, [1, 700, 130, 64, 333], [1, 260, 130, 0, 17], 32, 8, 128, 16),
    "ragged_d64_g2_bs32": (22, [45, 300, 97], [45, 120, 3], 8, 4, 64, 32),
    "g16_d128_bs64": (23, [200, 81], [150, 81], 16, 1, 128, 64),
    "mha_d64": (24, [129, 16, 17], [65, 16, 1], 4, 4, 64, 16),
}


@pytest.mark.parametrize("name", sorted(VARLEN_CASES))
def test_varlen_small_cases_all_rows(pa, name):
    seed, seq, ql, hq, hkv, hd, bs = VARLEN_CASES[name]
    b = workloads.make_paged_batch(name, seed, seq, ql, hq, hkv, hd, bs)
    d = Dev(pa, b)
    out, lse = _varlen(pa, d)
    ref_o, ref_l = oracle.paged_attention(b.q, d.ref_pool(), b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    assert_out_close(out, ref_o, name)
    assert_lse_close(lse, ref_l, name)
    assert pa.pa_get_device_error() == 0


def tile_boundary_rows(b, rows_per_tile, frac=0.01, seed=99):
    """Row mask of a full-size varlen batch: in every request, the first and
    last query row of each Q tile of the kernel (tile t holds query rows
    [t * rows_per_tile, (t + 1) * rows_per_tile) of the request), plus a
    random ``frac`` of all rows."""
    rng = np.random.default_rng(seed)
    mask = np.zeros(b.num_tokens, np.uint8)
    for i in range(b.num_seqs):
        a, e = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
        if e == a:
            continue
        starts = np.arange(a, e, rows_per_tile)
        mask[starts] = 1
        mask[np.minimum(starts + rows_per_tile - 1, e - 1)] = 1
    mask[rng.choice(b.num_tokens, max(1, int(frac * b.num_tokens)), replace=False)] = 1
    return mask


def test_varlen_chunked_prefill_full_size_sampled(pa):
    """The full chunked-prefill batch in the launch the bench times: every
    Q tile's first and last row (a tile is 128 packed (row, head) pairs, i.e.
    32 query rows at 4 q heads per kv head) of every request, plus 1 % random
    rows, all 32 heads."""
    b = workloads.chunked_prefill()
    d = Dev(pa, b, poison=False)
    out, lse = _varlen(pa, d)
    mask = tile_boundary_rows(b, 128 // (b.num_q_heads // b.num_kv_heads))
    ref_o, ref_l = oracle.paged_attention(b.q, d.ref_pool(), b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, row_mask=mask)
    rows = mask.astype(bool)
    assert rows.sum() > 1000
    assert_out_close(out[rows], ref_o[rows], "chunked prefill out")
    assert_lse_close(lse[rows], ref_l[rows], "chunked prefill lse")
    # Properties that hold for every row: finite outputs and LSE.
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------------------
# Split-KV decode + LSE merge
# ---------------------------------------------------------------------------

def _decode(pa, d, S):
    b = d.b
    N, hq = b.num_seqs, b.num_q_heads
    ws = pa.decode_workspace(N, hq, S, b.head_size)
    q = d.q.view(N, hq, b.head_size)
    out, lse = pa.pa_decode(q, d.pool, d.table, d.seq, b.scale, ws)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ws.cpu().numpy()


def test_decode_gqa_workload_all_requests(pa):
    b = workloads.gqa_decode()
    d = Dev(pa, b)
    pool = d.ref_pool()
    ref_o, ref_l = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    sms = pa.pa_device_sm_count()
    S_page = pa.pa_num_kv_splits(int(b.seq_lens.max()), sms)
    S_plan = pa.pa_decode_num_kv_splits(b.num_seqs, b.num_kv_heads, int(b.seq_lens.max()), sms)
    for S in sorted({S_page, S_plan, 1, 37}):
        out, lse, ws = _decode(pa, d, S)
        assert_out_close(out, ref_o, f"gqa decode S={S}")
        assert_lse_close(lse, ref_l, f"gqa decode lse S={S}")
        if S == S_page:
            part = oracle.split_partials(b.q, pool, b.block_table, b.seq_lens, b.scale, S)
            assert_lse_close(ws[..., -1], part[..., -1], "split lse")
            empty = np.isneginf(part[..., -1])
            assert not ws[..., :-1][empty].any()
            assert_out_close(ws[..., :-1][~empty], part[..., :-1][~empty], "split partial o")
    assert pa.pa_get_device_error() == 0


def test_decode_edge_cases(pa):
    # seq_len 0 (o = 0, lse = -inf), 1, a block boundary, ragged tails,
    # the largest supported group (16 q heads per kv head), block size 32.
    seq = [0, 1, 15, 16, 17, 31, 33, 250]
    b = workloads.make_paged_batch("edge", 31, seq, [0] * len(seq), 32, 2, 128, 32)
    d = Dev(pa, b)
    q = workloads.randn_bf16(np.random.default_rng(5), (len(seq), 32, 128))
    d.q = to_dev_bf16(q)
    # The oracle's decode: one split per request, merged (seq_len 0 allowed).
    part = oracle.split_partials(q, d.ref_pool(), b.block_table, np.asarray(seq, np.int32),
                                 b.scale, 1)
    ref_o, ref_l = oracle.lse_merge(part)
    for S in (1, 3, 16):
        out, lse, _ = _decode(pa, d, S)
        assert_out_close(out, ref_o, f"edge S={S}")
        assert_lse_close(lse, ref_l, f"edge lse S={S}")
    assert np.isneginf(lse[0]).all() and not out[0].any()
    assert pa.pa_get_device_error() == 0


def test_decode_d64(pa):
    b = workloads.make_paged_batch("d64", 32, [100, 517, 64], [1, 1, 1], 8, 2, 64, 16)
    d = Dev(pa, b)
    ref_o, ref_l = oracle.paged_attention(b.q, d.ref_pool(), b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    out, lse, _ = _decode(pa, d, 5)
    assert_out_close(out, ref_o, "d64 decode")
    assert_lse_close(lse, ref_l, "d64 decode lse")


def test_decode_long_context_full_size_sampled(pa):
    b = workloads.long_decode()
    d = Dev(pa, b, poison=False)
    # The long-context workload fixes S = min(ceil(seq / 512), 2 * SMs).
    sms = pa.pa_device_sm_count()
    S = min(math.ceil(131072 / 512), 2 * sms)
    assert pa.pa_num_kv_splits(131072, sms) == S
    out, lse, _ = _decode(pa, d, S)
    # The step's 8 new tokens landed bit-exactly.
    s = b.slot_mapping
    got_k = bf16_bits(d.pool[torch.from_numpy(s // 16), 0, torch.from_numpy(s % 16)])
    assert np.array_equal(got_k, b.key)
    got_v = bf16_bits(d.pool[torch.from_numpy(s // 16), 1, torch.from_numpy(s % 16)])
    assert np.array_equal(got_v, b.value)
    # Every request against the oracle.
    pool = d.ref_pool()
    ref_o, ref_l = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    assert_out_close(out, ref_o, "long decode out")
    assert_lse_close(lse, ref_l, "long decode lse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert pa.pa_get_device_error() == 0


# (S, dv): one split, the warp-per-head merge at and below its split limits
# (8 and 16 at dv 128, 32 at dv 64) and one past them, a group of splits that
# fills a warp and one past it, hundreds of splits; value widths of the
# standard pool and of MLA.
@pytest.mark.parametrize("S,dv", [(13, 128), (1, 64), (8, 128), (16, 128), (17, 128), (32, 64),
                                  (33, 64), (32, 512), (33, 128), (300, 64)])
def test_lse_merge_random_partials(pa, S, dv):
    rng = np.random.default_rng(41 + S)
    N, H = 5, 7                                   # 35 heads: not a multiple of 4
    part = rng.standard_normal((N, H, S, dv + 1)).astype(np.float32)
    part[..., -1] *= 4.0
    part[0, 0, S // 4:, -1] = -np.inf             # some empty splits (all but the first, S = 1..3)
    part[1, 2, :, -1] = -np.inf                   # all empty
    part[..., :-1][np.isneginf(part[..., -1])] = 0.0
    ws = torch.from_numpy(part).cuda()
    out, lse = pa.pa_lse_merge(ws)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.lse_merge(part.astype(np.float64))
    assert_out_close(bf16_to_f64(out), ref_o, "merge")
    assert_lse_close(lse.cpu().numpy(), ref_l, "merge lse", atol=1e-5)


def test_invalid_block_id_is_flagged_not_read(pa):
    b = workloads.make_paged_batch("badblk", 33, [40, 64], [1, 1], 8, 2, 128, 16)
    table = b.block_table.copy()
    table[0, 1] = b.num_blocks + 1000
    d = Dev(pa, b)
    d.table = to_dev(table, torch.int32)
    ref_o, ref_l = oracle.paged_attention(b.q, d.ref_pool(), b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    out, lse, _ = _decode(pa, d, 2)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    assert_out_close(out[1], ref_o[1], "untouched request")
    o2, l2 = _varlen(pa, d)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    assert_out_close(o2[1], ref_o[1], "untouched request (varlen)")


# ---------------------------------------------------------------------------
# MLA latent decode
# ---------------------------------------------------------------------------

def _poison_mla(b):
    pool = b.pool.copy()
    used = np.zeros((b.num_blocks, b.block_size), bool)
    for i in range(b.batch):
        pos = np.arange(int(b.seq_lens[i]))
        used[b.block_table[i, pos // b.block_size], pos % b.block_size] = True
    pool[~used] = BF16_NAN
    return pool


def _mla(pa, b, S, pool):
    d_pool = to_dev_bf16(pool)
    q = to_dev_bf16(b.q)
    ws = pa.decode_workspace(b.batch, b.num_heads, S, b.kv_lora_rank)
    out, lse = pa.pa_mla_decode(q, d_pool, to_dev(b.block_table, torch.int32),
                                to_dev(b.seq_lens, torch.int32), b.scale, ws)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


def test_mla_small_all_heads(pa):
    b = workloads.make_mla_batch("mla_small", 51, [1, 63, 64, 65, 700, 0], 128,
                                 scale=1.0 / math.sqrt(192.0))
    pool = _poison_mla(b)
    ref_o, ref_l = oracle.mla_decode(b.q, pool, b.block_table, b.seq_lens, b.scale)
    for S in (1, 3):
        out, lse = _mla(pa, b, S, pool)
        assert_out_close(out, ref_o, f"mla S={S}")
        assert_lse_close(lse, ref_l, f"mla lse S={S}")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("heads,bs", [(64, 32), (256, 128), (128, 32)])
def test_mla_head_groups_and_block_sizes(pa, heads, bs):
    """A head count below one 128-head group (spare rows computed, never
    stored), two head groups, and blocks of 32 and 128 tokens (a 64-token
    tile spans two blocks, or half a block); unused pool slots hold NaN."""
    b = workloads.make_mla_batch(f"mla_h{heads}_bs{bs}", 52, [1, 33, 64, 130, 257, 0], heads,
                                 block_size=bs, scale=1.0 / math.sqrt(192.0))
    pool = _poison_mla(b)
    ref_o, ref_l = oracle.mla_decode(b.q, pool, b.block_table, b.seq_lens, b.scale)
    for S in (1, 2):
        out, lse = _mla(pa, b, S, pool)
        assert_out_close(out, ref_o, f"mla H={heads} bs={bs} S={S}")
        assert_lse_close(lse, ref_l, f"mla lse H={heads} bs={bs} S={S}")
    assert pa.pa_get_device_error() == 0


def test_mla_workload_full_size_sampled(pa):
    """The full DeepSeek-V3-shape batch: 20 requests -- the 4 longest, the 4
    shortest (the first and last the longest-first dispatch hands out) and
    12 drawn at random -- all heads, one and two splits."""
    b = workloads.mla_decode()
    order = np.argsort(b.seq_lens, kind="stable")
    pick = set(order[:4].tolist()) | set(order[-4:].tolist())
    rest = np.setdiff1d(np.arange(b.batch), sorted(pick))
    pick |= set(np.random.default_rng(98).choice(rest, 12, replace=False).tolist())
    mask = np.zeros(b.batch, np.uint8)
    mask[sorted(pick)] = 1
    assert mask.sum() == 20
    ref_o, ref_l = oracle.mla_decode(b.q, b.pool, b.block_table, b.seq_lens, b.scale,
                                     req_mask=mask)
    rows = mask.astype(bool)
    # One split (the output written by the stage-1 kernel) and two (the merge).
    for S in (1, 2):
        out, lse = _mla(pa, b, S, b.pool)
        assert_out_close(out[rows], ref_o[rows], f"mla out S={S}")
        assert_lse_close(lse[rows], ref_l[rows], f"mla lse S={S}")
        assert np.isfinite(out).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------------------
# MLA cache write
# ---------------------------------------------------------------------------

def test_mla_cache_write_then_decode(pa):
    """The step's new latent rows land bit-exactly (whole pool compared), and
    the MLA decode over the written pool matches the oracle's."""
    b = workloads.make_mla_batch("mla_write", 53, [1, 63, 64, 65, 700, 0], 128,
                                 scale=1.0 / math.sqrt(192.0))
    kv_c, k_pe, slots = workloads.mla_new_tokens(b)
    pool = _poison_mla(b)
    d_pool = to_dev_bf16(pool)
    pa.pa_mla_cache_write(to_dev_bf16(kv_c), to_dev_bf16(k_pe), d_pool,
                          to_dev(slots, torch.int64))
    ref_pool = oracle.mla_cache_write(kv_c, k_pe, pool, slots, b.block_size)
    assert np.array_equal(bf16_bits(d_pool), ref_pool)
    assert pa.pa_get_device_error() == 0
    ref_o, ref_l = oracle.mla_decode(b.q, ref_pool, b.block_table, b.seq_lens, b.scale)
    ws = pa.decode_workspace(b.batch, b.num_heads, 2, b.kv_lora_rank)
    out, lse = pa.pa_mla_decode(to_dev_bf16(b.q), d_pool, to_dev(b.block_table, torch.int32),
                                to_dev(b.seq_lens, torch.int32), b.scale, ws)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o, "mla after write")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_l, "mla lse after write")


def test_mla_cache_write_skip_out_of_range_and_full_workload(pa):
    b = workloads.mla_decode()
    kv_c, k_pe, slots = workloads.mla_new_tokens(b)
    slots = slots.copy()
    slots[5] = -1
    slots[9] = b.num_blocks * b.block_size + 7      # outside the pool: flagged, not written
    d_pool = to_dev_bf16(b.pool)
    pa.pa_mla_cache_write(to_dev_bf16(kv_c), to_dev_bf16(k_pe), d_pool,
                          to_dev(slots, torch.int64))
    assert pa.pa_get_device_error() == pa.PA_DEVERR_SLOT
    keep = slots.copy()
    keep[9] = -1
    ref_pool = oracle.mla_cache_write(kv_c, k_pe, b.pool, keep, b.block_size)
    assert np.array_equal(bf16_bits(d_pool), ref_pool)
    assert pa.pa_get_device_error() == 0
