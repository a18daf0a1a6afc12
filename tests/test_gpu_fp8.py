"""GPU parity of the fp8 (e4m3) KV cache, through the C ABI, against the fp64
oracle on the same seeded inputs.

The quantising cache write must produce the oracle's codes bit for bit (NaN
inputs: any NaN code).  Split-KV decode over an fp8 pool must meet the
tolerances of ``tests/parity.py`` against the oracle's split partials over the
dequantised pool (code value times k_scale or v_scale, in fp64).

Unused pool slots and the unused tail of every request's last block hold the
NaN code 0x7F, so a kernel that read anything outside a request's first
seq_len tokens would produce NaN and fail.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import (assert_lse_close, assert_out_close, bf16_to_f64, to_dev,
                          to_dev_bf16)

pytestmark = pytest.mark.gpu

KS, VS = workloads.FP8_K_SCALE, workloads.FP8_V_SCALE
NAN_CODE = np.uint8(0x7F)


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


def _used(b):
    used = np.zeros((b.num_blocks, b.block_size), bool)
    for i in range(b.num_seqs):
        n = int(b.seq_lens[i])
        if n == 0:
            continue
        pos = np.arange(n)
        used[b.block_table[i, pos // b.block_size], pos % b.block_size] = True
    return used


class Dev8:
    """A batch with an fp8 pool on the device, after the step's quantising
    cache write."""

    def __init__(self, pa, b, poison=True, ks=KS, vs=VS, as_float8=False):
        self.b, self.ks, self.vs = b, ks, vs
        pool = workloads.fp8_pool(b)
        if poison:
            pool.transpose(0, 2, 1, 3, 4)[~_used(b)] = NAN_CODE
        self.host_pool_before = pool
        self.pool = torch.from_numpy(pool.copy()).cuda()
        if as_float8:
            self.pool = self.pool.view(torch.float8_e4m3fn)
        self.q = to_dev_bf16(b.q)
        self.key = to_dev_bf16(b.key)
        self.value = to_dev_bf16(b.value)
        self.slots = to_dev(b.slot_mapping, torch.int64)
        self.table = to_dev(b.block_table, torch.int32)
        self.seq = to_dev(b.seq_lens, torch.int32)
        pa.pa_reshape_and_cache_fp8(self.key, self.value, self.pool, self.slots, ks, vs)

    def codes(self):
        return self.pool.view(torch.uint8).cpu().numpy()

    def ref_pool(self):
        b = self.b
        return oracle.reshape_and_cache_fp8(b.key, b.value, self.host_pool_before,
                                            b.slot_mapping, b.block_size, self.ks, self.vs)

    def decode(self, pa, S, q=None):
        """Both split-KV stages over the fp8 pool for one query per request
        (default: each request's last query row)."""
        b = self.b
        N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
        ws = pa.decode_workspace(N, hq, S, d)
        q = to_dev_bf16(_decode_q(b)) if q is None else q
        out, lse = pa.pa_decode_fp8(q, self.pool, self.table, self.seq, b.scale, self.ks,
                                    self.vs, ws)
        torch.cuda.synchronize()
        return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ws.cpu().numpy()


# ---------------------------------------------------------------------------
# Quantising cache write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("make", [workloads.tiny_paged, workloads.gqa_decode,
                                  workloads.chunked_prefill],
                         ids=["tiny", "gqa_decode", "chunked_prefill"])
def test_fp8_cache_write_bit_exact(pa, make):
    b = make(with_pool=False) if make is not workloads.tiny_paged else make()
    d = Dev8(pa, b)
    assert np.array_equal(d.codes(), d.ref_pool())
    assert pa.pa_get_device_error() == 0


def _special_values():
    """bf16 bit patterns for the quantiser's edge cases at scale 1: exact codes,
    ties between codes (which go to the even code), the subnormal range, the
    saturation boundary, infinities, signed zeros."""
    f = np.array([
        0.0, -0.0, 1.0, -1.0, 1.0625, 1.1875, -1.0625, 3.25,            # ties at [1, 2)
        2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -11, -2.0 ** -10,  # subnormal grid
        2.0 ** -6, 2.0 ** -7 + 2.0 ** -10,                               # normal/subnormal edge
        448.0, -448.0, 464.0, 480.0, 500.0, 1e4, -3e38,                  # saturation
        np.inf, -np.inf, 1e-30, -1e-30, 240.0, 232.0, 0.013671875, 17.0,
    ], np.float32)
    return workloads.f32_to_bf16_bits(f)


@pytest.mark.parametrize("scales", [(1.0, 1.0), (KS, VS), (0.5, 3.0)])
def test_fp8_cache_write_edge_values(pa, scales):
    ks, vs = scales
    b = workloads.make_paged_batch("fp8_edge", 40, [64, 16], [64, 16], 4, 2, 64, 16,
                                   with_pool=False)
    key = b.key.copy()
    value = b.value.copy()
    sv = _special_values()
    key.reshape(-1)[:sv.size] = sv
    value.reshape(-1)[-sv.size:] = sv[::-1]
    b.key, b.value = key, value
    d = Dev8(pa, b, ks=ks, vs=vs)
    assert np.array_equal(d.codes(), d.ref_pool())


def test_fp8_cache_write_nan_input_gives_a_nan_code(pa):
    b = workloads.make_paged_batch("fp8_nan", 41, [16], [16], 4, 2, 64, 16, with_pool=False)
    key = b.key.copy()
    key[3, 1, 5] = 0x7FC0                   # +NaN
    key[7, 0, 0] = 0xFFC0                   # -NaN
    b.key = key
    d = Dev8(pa, b, poison=False)
    got, ref = d.codes(), d.ref_pool()
    nan_at = np.isin(got, [0x7F, 0xFF])
    assert np.array_equal(nan_at, np.isin(ref, [0x7F, 0xFF]))
    assert nan_at.sum() == 2
    assert np.array_equal(got[~nan_at], ref[~nan_at])


def test_fp8_cache_write_skip_and_out_of_range(pa):
    b = workloads.tiny_paged()
    slots = b.slot_mapping.copy()
    slots[1] = -1
    slots[3] = b.num_blocks * b.block_size          # first slot past the pool
    pool = workloads.fp8_pool(b)
    d_pool = torch.from_numpy(pool.copy()).cuda()
    pa.pa_reshape_and_cache_fp8(to_dev_bf16(b.key), to_dev_bf16(b.value), d_pool,
                                to_dev(slots, torch.int64), KS, VS)
    assert pa.pa_get_device_error() == pa.PA_DEVERR_SLOT
    keep = slots.copy()
    keep[3] = -1
    ref = oracle.reshape_and_cache_fp8(b.key, b.value, pool, keep, b.block_size, KS, VS)
    assert np.array_equal(d_pool.cpu().numpy(), ref)
    assert pa.pa_get_device_error() == 0


def test_fp8_pool_as_float8_dtype(pa):
    b = workloads.tiny_paged()
    d = Dev8(pa, b, as_float8=True)
    assert d.pool.dtype == torch.float8_e4m3fn
    assert np.array_equal(d.codes(), d.ref_pool())
    out, lse, _ = d.decode(pa, 2)
    part = oracle.split_partials_fp8(_decode_q(b), d.ref_pool(), b.block_table, b.seq_lens,
                                     b.scale, KS, VS, 1)
    ref_o, ref_l = oracle.lse_merge(part)
    assert_out_close(out, ref_o, "float8 pool decode")
    assert_lse_close(lse, ref_l, "float8 pool decode lse")


# ---------------------------------------------------------------------------
# Split-KV decode over the fp8 pool
# ---------------------------------------------------------------------------

def _decode_q(b):
    """One decode query per request: the last query row of each request."""
    last = b.query_start_loc[1:] - 1
    return b.q[last]


def test_fp8_decode_gqa_workload_all_requests(pa):
    b = workloads.gqa_decode(with_pool=False)
    d = Dev8(pa, b)
    pool = d.ref_pool()
    assert np.array_equal(d.codes(), pool)
    q = _decode_q(b)
    sms = pa.pa_device_sm_count()
    S_page = pa.pa_num_kv_splits(int(b.seq_lens.max()), sms)
    ref_o = ref_l = None
    for S in sorted({S_page, 1, 37}):
        part = oracle.split_partials_fp8(q, pool, b.block_table, b.seq_lens, b.scale, KS, VS, S)
        if ref_o is None:
            ref_o, ref_l = oracle.lse_merge(part)
        out, lse, ws = d.decode(pa, S)
        assert_out_close(out, ref_o, f"fp8 gqa decode S={S}")
        assert_lse_close(lse, ref_l, f"fp8 gqa decode lse S={S}")
        assert_lse_close(ws[..., -1], part[..., -1], f"fp8 split lse S={S}")
        empty = np.isneginf(part[..., -1])
        assert not ws[..., :-1][empty].any()
        assert_out_close(ws[..., :-1][~empty], part[..., :-1][~empty], f"fp8 split o S={S}")
    assert pa.pa_get_device_error() == 0


def test_fp8_decode_long_context_full_size_sampled(pa):
    """The long-context batch (8 x 131072 tokens, 64 q / 8 kv heads) over an
    fp8 pool at the split count the bench times: the step's 8 new rows are
    quantised bit-exactly, and every request matches the oracle, which runs
    on one request's blocks at a time (the whole pool in fp64 would take
    17 GB)."""
    b = workloads.long_decode(with_pool=False)
    d = Dev8(pa, b, poison=False)
    sms = pa.pa_device_sm_count()
    S = min(math.ceil(131072 / 512), 2 * sms)
    assert pa.pa_num_kv_splits(131072, sms) == S
    out, lse, _ = d.decode(pa, S)
    bs = b.block_size
    s = b.slot_mapping
    # Expected codes of the new rows: the oracle's write into a small pool,
    # one block per request, at the same offsets.
    small = np.zeros((b.num_seqs, 2, bs, b.num_kv_heads, b.head_size), np.uint8)
    small = oracle.reshape_and_cache_fp8(b.key, b.value, small,
                                         np.arange(b.num_seqs) * bs + s % bs, bs, KS, VS)
    rows = d.pool.view(torch.uint8)[torch.from_numpy(s // bs).cuda(), :,
                                    torch.from_numpy(s % bs).cuda()].cpu().numpy()
    assert np.array_equal(rows, small[np.arange(b.num_seqs), :, s % bs])
    q = _decode_q(b)
    for r in range(b.num_seqs):
        n = int(b.seq_lens[r])
        blocks = b.block_table[r, :(n + bs - 1) // bs]
        sub = oracle.reshape_and_cache_fp8(b.key[r:r + 1], b.value[r:r + 1],
                                           d.host_pool_before[blocks], np.array([n - 1]), bs,
                                           KS, VS)
        table = np.arange(len(blocks), dtype=np.int32)[None, :]
        part = oracle.split_partials_fp8(q[r:r + 1], sub, table, b.seq_lens[r:r + 1], b.scale,
                                         KS, VS, 1)
        ref_o, ref_l = oracle.lse_merge(part)
        assert_out_close(out[r:r + 1], ref_o, f"fp8 long decode out, request {r}")
        assert_lse_close(lse[r:r + 1], ref_l, f"fp8 long decode lse, request {r}")
        del sub, part
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert pa.pa_get_device_error() == 0


def test_fp8_decode_edge_cases(pa):
    # seq_len 0 (o = 0, lse = -inf), 1, a block boundary, ragged tails, the
    # largest supported group (16 q heads per kv head), block size 32.
    seq = [0, 1, 15, 16, 17, 31, 33, 250]
    b = workloads.make_paged_batch("fp8_edge_dec", 31, seq, [0] * len(seq), 32, 2, 128, 32,
                                   with_pool=False)
    d = Dev8(pa, b)
    q = workloads.randn_bf16(np.random.default_rng(5), (len(seq), 32, 128))
    part = oracle.split_partials_fp8(q, d.ref_pool(), b.block_table, b.seq_lens, b.scale, KS,
                                     VS, 1)
    ref_o, ref_l = oracle.lse_merge(part)
    for S in (1, 3, 16):
        out, lse, _ = d.decode(pa, S, q=to_dev_bf16(q))
        assert_out_close(out, ref_o, f"fp8 edge S={S}")
        assert_lse_close(lse, ref_l, f"fp8 edge lse S={S}")
    assert np.isneginf(lse[0]).all() and not out[0].any()
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("group", [1, 4, 7])
def test_fp8_decode_d64_and_groups(pa, group):
    b = workloads.make_paged_batch(f"fp8_d64_g{group}", 32 + group, [100, 517, 64, 1000],
                                   [1, 1, 1, 1], 2 * group, 2, 64, 16, with_pool=False)
    d = Dev8(pa, b)
    part = oracle.split_partials_fp8(b.q, d.ref_pool(), b.block_table, b.seq_lens, b.scale, KS,
                                     VS, 1)
    ref_o, ref_l = oracle.lse_merge(part)
    out, lse, _ = d.decode(pa, 5)
    assert_out_close(out, ref_o, f"fp8 d64 decode g={group}")
    assert_lse_close(lse, ref_l, f"fp8 d64 decode lse g={group}")


def test_fp8_decode_max_value_codes(pa):
    # Every K and V entry at the largest finite code (+-448): the largest
    # products the f16 operands carry.
    b = workloads.make_paged_batch("fp8_max", 42, [48, 200], [1, 1], 8, 2, 128, 16,
                                   with_pool=False)
    d = Dev8(pa, b, poison=False, ks=0.004, vs=0.01)
    rng = np.random.default_rng(9)
    sign = rng.integers(0, 2, size=d.host_pool_before.shape).astype(np.uint8) << 7
    codes = (sign | np.uint8(0x7E)).astype(np.uint8)
    d.host_pool_before = codes
    d.pool = torch.from_numpy(codes.copy()).cuda()
    part = oracle.split_partials_fp8(b.q, codes, b.block_table, b.seq_lens, b.scale, 0.004, 0.01,
                                     1)
    ref_o, ref_l = oracle.lse_merge(part)
    out, lse, _ = d.decode(pa, 3)
    assert_out_close(out, ref_o, "fp8 max codes")
    assert_lse_close(lse, ref_l, "fp8 max codes lse")


def test_fp8_invalid_block_id_is_flagged_not_read(pa):
    b = workloads.make_paged_batch("fp8_badblk", 33, [40, 64], [1, 1], 8, 2, 128, 16,
                                   with_pool=False)
    d = Dev8(pa, b)
    part = oracle.split_partials_fp8(b.q, d.ref_pool(), b.block_table, b.seq_lens, b.scale, KS,
                                     VS, 1)
    ref_o, _ = oracle.lse_merge(part)
    table = b.block_table.copy()
    table[0, 1] = b.num_blocks + 1000
    d.table = to_dev(table, torch.int32)
    out, _, _ = d.decode(pa, 2)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_BLOCK_ID
    assert_out_close(out[1], ref_o[1], "untouched request")
    assert np.isfinite(out[0]).all()
