"""GPU parity of the sliding-window and cascade (shared-prefix) variants of
varlen paged attention, through the C ABI, against the fp64 oracle.

Cascade attention must give the result of plain attention over each
request's whole sequence (the oracle's paged_attention); its prefix pass,
suffix pass and merge are checked together and, for the split partials,
against the oracle's split reference.  Unused pool slots hold NaN as in
``test_gpu_parity.py``.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import assert_lse_close, assert_out_close, bf16_to_f64
from tests.test_gpu_parity import Dev

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


def _np(out, lse):
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------------------
# Sliding window
# ---------------------------------------------------------------------------

WINDOW_CASES = {
    # name: (seed, seq_lens, query_lens, Hq, Hkv, d, bs, windows)
    "ragged_d128_g4": (31, [1, 700, 130, 64, 333], [1, 260, 130, 0, 17], 32, 8, 128, 16,
                       [1, 7, 128, 129, 300]),
    "d64_g2_bs32": (32, [45, 300, 97], [45, 120, 3], 8, 4, 64, 32, [16, 33, 1000]),
    "g16_long_rows": (33, [900, 81], [700, 81], 16, 1, 128, 64, [200, 255, 256, 257]),
}


@pytest.mark.parametrize("name", sorted(WINDOW_CASES))
def test_window_all_rows(pa, name):
    seed, seq, ql, hq, hkv, hd, bs, windows = WINDOW_CASES[name]
    b = workloads.make_paged_batch(name, seed, seq, ql, hq, hkv, hd, bs)
    d = Dev(pa, b)
    pool = d.ref_pool()
    mq = int(b.query_lens.max())
    for W in windows:
        out, lse = _np(*pa.pa_varlen_fwd_window(d.q, d.pool, d.table, d.qsl, d.seq, mq, b.scale,
                                                W))
        ref_o, ref_l = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                              b.seq_lens, b.scale, window=W)
        assert_out_close(out, ref_o, f"{name} W={W}")
        assert_lse_close(lse, ref_l, f"{name} W={W} lse")
    assert pa.pa_get_device_error() == 0


def test_window_wider_than_every_sequence_equals_causal(pa):
    name = "ragged_d128_g4"
    seed, seq, ql, hq, hkv, hd, bs, _ = WINDOW_CASES[name]
    b = workloads.make_paged_batch(name, seed, seq, ql, hq, hkv, hd, bs)
    d = Dev(pa, b)
    mq = int(b.query_lens.max())
    o1, l1 = pa.pa_varlen_fwd(d.q, d.pool, d.table, d.qsl, d.seq, mq, b.scale)
    o2, l2 = pa.pa_varlen_fwd_window(d.q, d.pool, d.table, d.qsl, d.seq, mq, b.scale, 100000)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_chunked_prefill_full_size_sampled(pa):
    b = workloads.chunked_prefill()
    d = Dev(pa, b, poison=False)
    W = 1024
    out, lse = _np(*pa.pa_varlen_fwd_window(d.q, d.pool, d.table, d.qsl, d.seq,
                                            int(b.query_lens.max()), b.scale, W))
    rng = np.random.default_rng(98)
    mask = np.zeros(b.num_tokens, np.uint8)
    for i in range(b.num_seqs):
        a, e = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
        mask[[a, e - 1]] = 1
        mask[rng.integers(a, e, size=3)] = 1
    ref_o, ref_l = oracle.paged_attention(b.q, d.ref_pool(), b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, row_mask=mask, window=W)
    rows = mask.astype(bool)
    assert_out_close(out[rows], ref_o[rows], "windowed chunked prefill out")
    assert_lse_close(lse[rows], ref_l[rows], "windowed chunked prefill lse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------------------
# Cascade attention
# ---------------------------------------------------------------------------

def _cascade(pa, d, P, S1, S2=1, causal=True):
    b = d.b
    ws = pa.cascade_workspace(b.num_tokens, b.num_q_heads, S1, S2, b.head_size)
    out, lse = pa.pa_cascade_fwd(d.q, d.pool, d.table, d.qsl, d.seq, int(b.query_lens.max()), P,
                                 b.scale, ws, S1, causal=causal)
    o, l = _np(out, lse)
    return o, l, ws.cpu().numpy()


CASCADE_CASES = {
    # name: (seed, prefix_blocks, suffix_lens, query_lens, Hq, Hkv, d, bs)
    "decode_d128_g4": (41, 20, [17, 300, 1, 64, 129], [1, 1, 1, 1, 1], 32, 8, 128, 16),
    "prefill_d128_g4": (42, 9, [200, 31, 130], [150, 31, 2], 32, 8, 128, 16),
    "d64_g2_bs32": (43, 5, [45, 300, 97], [45, 120, 3], 8, 4, 64, 32),
    "g16_bs64": (44, 3, [81, 200], [81, 20], 16, 1, 128, 64),
}


@pytest.mark.parametrize("name", sorted(CASCADE_CASES))
def test_cascade_equals_plain_attention(pa, name):
    seed, P, suf, ql, hq, hkv, hd, bs = CASCADE_CASES[name]
    b = workloads.make_shared_prefix_batch(name, seed, P, suf, ql, hq, hkv, hd, bs)
    d = Dev(pa, b)
    pool = d.ref_pool()
    ref_o, ref_l = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    for S1, S2 in ((1, 1), (3, 1), (2, 5)):
        out, lse, ws = _cascade(pa, d, P, S1, S2)
        assert_out_close(out, ref_o, f"{name} cascade S1={S1} S2={S2}")
        assert_lse_close(lse, ref_l, f"{name} cascade S1={S1} S2={S2} lse")
    assert pa.pa_get_device_error() == 0


def test_cascade_partials_match_the_oracle(pa):
    # Pass 1 slots = the oracle's split partials of every row against the
    # prefix alone (non-causal: one request of all rows with the prefix as its
    # context); pass 2 slot = the oracle's attention over each request's own
    # tokens after the prefix.
    seed, P, suf, ql, hq, hkv, hd, bs = CASCADE_CASES["prefill_d128_g4"]
    b = workloads.make_shared_prefix_batch("partials", seed, P, suf, ql, hq, hkv, hd, bs)
    d = Dev(pa, b)
    pool = d.ref_pool()
    S1 = 2
    _, _, ws = _cascade(pa, d, P, S1)
    T = b.num_tokens
    prefix = P * bs
    # The prefix as one request of all T rows, non-causal, split like pass 1
    # (chunks of 128-token multiples: ceil(ceil(prefix / S1) / 128) * 128).
    chunk = -(-(-(-prefix // S1)) // 128) * 128
    for s in range(S1):
        a, e = s * chunk, (prefix if s == S1 - 1 else min(prefix, (s + 1) * chunk))
        a = min(a, prefix)
        n = e - a
        if n == 0:
            assert np.isneginf(ws[:, :, s, -1]).all() and not ws[:, :, s, :-1].any()
            continue
        # Every row as a one-query request over tokens [a, e) of the shared
        # prefix (blocks a/bs .. of table row 0), no mask.
        table = b.block_table[:1, a // bs:(e + bs - 1) // bs]
        ref_o, ref_l = oracle.paged_attention(b.q, pool, np.repeat(table, T, axis=0),
                                              np.arange(T + 1, dtype=np.int32),
                                              np.full(T, n, np.int32), b.scale, causal=False)
        assert_out_close(ws[:, :, s, :-1], ref_o, f"prefix partial {s}")
        assert_lse_close(ws[:, :, s, -1], ref_l, f"prefix partial {s} lse")
    # Pass 2: each request over its own suffix, causal.
    suf_table = np.full_like(b.block_table, -1)
    suf_table[:, :b.block_table.shape[1] - P] = b.block_table[:, P:]
    ref_o, ref_l = oracle.paged_attention(b.q, pool, suf_table, b.query_start_loc,
                                          b.seq_lens - prefix, b.scale)
    assert_out_close(ws[:, :, S1, :-1], ref_o, "suffix partial")
    assert_lse_close(ws[:, :, S1, -1], ref_l, "suffix partial lse")


def test_cascade_non_causal_and_no_prefix(pa):
    seed, P, suf, ql, hq, hkv, hd, bs = CASCADE_CASES["prefill_d128_g4"]
    b = workloads.make_shared_prefix_batch("nc", seed, P, suf, ql, hq, hkv, hd, bs)
    d = Dev(pa, b)
    pool = d.ref_pool()
    ref_o, ref_l = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, causal=False)
    out, lse, _ = _cascade(pa, d, P, 2, 2, causal=False)
    assert_out_close(out, ref_o, "non-causal cascade")
    assert_lse_close(lse, ref_l, "non-causal cascade lse")
    # No shared prefix: the plain path.
    ref_o, ref_l = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    out, lse, _ = _cascade(pa, d, 0, 1)
    assert_out_close(out, ref_o, "cascade without prefix")
    assert_lse_close(lse, ref_l, "cascade without prefix lse")


def test_cascade_query_inside_prefix_is_flagged(pa):
    # A request whose new tokens start inside the shared blocks breaks the
    # precondition: the call flags it (and its rows are not checked).
    b = workloads.make_shared_prefix_batch("inside", 45, 4, [10, 40], [2, 2], 8, 2, 128, 16)
    d = Dev(pa, b)
    assert pa.pa_get_device_error() == 0
    # Two queries per request, so the varlen suffix pass (which checks) runs.
    ws = pa.cascade_workspace(b.num_tokens, 8, 1, 1, 128)
    pa.pa_cascade_fwd(d.q, d.pool, d.table, d.qsl, d.seq, int(b.query_lens.max()), 5, b.scale,
                      ws, 1)   # 5 > 4 shared blocks
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.PA_DEVERR_LENGTH


def test_cascade_shared_prefix_decode_full_size_sampled(pa):
    b = workloads.shared_prefix_decode()
    d = Dev(pa, b, poison=False)
    P = 4096 // 16
    S1 = pa.pa_cascade_prefix_splits(b.num_tokens, b.num_q_heads, b.num_kv_heads, 4096)
    S2 = pa.pa_num_kv_splits(int(b.seq_lens.max()) - 4096)
    out, lse, _ = _cascade(pa, d, P, S1, S2)
    mask = np.zeros(b.num_tokens, np.uint8)
    mask[[0, 7, 31, 63]] = 1
    ref_o, ref_l = oracle.paged_attention(b.q, d.ref_pool(), b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, row_mask=mask)
    rows = mask.astype(bool)
    assert_out_close(out[rows], ref_o[rows], "shared-prefix decode out")
    assert_lse_close(lse[rows], ref_l[rows], "shared-prefix decode lse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert pa.pa_get_device_error() == 0
