"""The library at its maximum sizes, against the oracle.

* 65535 requests (the largest grid dimension the launches use for requests)
  in split-KV decode and in varlen attention, every row;
* 16384 splits (the largest the merge accepts) on a short batch: almost
  every split is empty and the merge must still give the unsplit result;
* an MLA batch of 600 requests, more than the 512 the MLA kernel ranks by
  length, so the pairs take requests in grid order.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import assert_lse_close, assert_out_close, bf16_to_f64, to_dev, to_dev_bf16

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


def _pool_after_write(pa, b):
    pool = to_dev_bf16(b.pool)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key), to_dev_bf16(b.value), pool,
                            to_dev(b.slot_mapping, torch.int64))
    return pool, oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)


def test_decode_and_varlen_with_65535_requests(pa):
    rng = np.random.default_rng(91)
    N = 65535
    seq = rng.integers(1, 40, size=N, endpoint=True)
    qlen = np.minimum(seq, rng.integers(1, 3, size=N, endpoint=True))
    b = workloads.make_paged_batch("max_requests", 91, seq, qlen, 8, 2, 64, 16)
    pool, ref_pool = _pool_after_write(pa, b)
    table = to_dev(b.block_table, torch.int32)
    seql = to_dev(b.seq_lens, torch.int32)
    # Varlen attention over every row of all 65535 requests.
    out, lse = pa.pa_varlen_fwd(to_dev_bf16(b.q), pool, table, to_dev(b.query_start_loc, torch.int32),
                                seql, int(b.query_lens.max()), b.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    assert_out_close(bf16_to_f64(out), ref_o, "varlen, 65535 requests")
    assert_lse_close(lse.cpu().numpy(), ref_l, "varlen lse, 65535 requests")
    # Split-KV decode of each request's last row (3 splits).
    last = b.query_start_loc[1:] - 1
    q = to_dev_bf16(b.q[last]).view(N, 8, 64)
    ws = pa.decode_workspace(N, 8, 3, 64)
    out, lse = pa.pa_decode(q, pool, table, seql, b.scale, ws)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o[last], "decode, 65535 requests")
    assert_lse_close(lse.cpu().numpy(), ref_l[last], "decode lse, 65535 requests")
    assert pa.pa_get_device_error() == 0


def test_decode_with_16384_splits(pa):
    b = workloads.make_paged_batch("max_splits", 92, [100, 5000, 1], [1, 1, 1], 8, 2, 128, 16)
    pool, ref_pool = _pool_after_write(pa, b)
    ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    q = to_dev_bf16(b.q).view(3, 8, 128)
    table, seql = to_dev(b.block_table, torch.int32), to_dev(b.seq_lens, torch.int32)
    for S in (16384, 1):
        ws = pa.decode_workspace(3, 8, S, 128)
        out, lse = pa.pa_decode(q, pool, table, seql, b.scale, ws)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out), ref_o, f"decode S={S}")
        assert_lse_close(lse.cpu().numpy(), ref_l, f"decode lse S={S}")
        if S > 1:
            # Every split past a request's end is empty: lse -inf, o = 0.
            part = ws.cpu().numpy()
            assert np.isneginf(part[0, :, 7:, -1]).all() and not part[0, :, 7:, :-1].any()
    assert pa.pa_get_device_error() == 0


def test_mla_batch_beyond_the_ranked_size(pa):
    rng = np.random.default_rng(93)
    B = 600                                      # > 512: pairs take requests in grid order
    seq = rng.integers(1, 80, size=B, endpoint=True)
    m = workloads.make_mla_batch("mla_600", 93, seq, 128, scale=1.0 / math.sqrt(192.0))
    ref_o, ref_l = oracle.mla_decode(m.q, m.pool, m.block_table, m.seq_lens, m.scale)
    for S in (1, 2):
        ws = pa.decode_workspace(B, 128, S, 512)
        out, lse = pa.pa_mla_decode(to_dev_bf16(m.q), to_dev_bf16(m.pool),
                                    to_dev(m.block_table, torch.int32),
                                    to_dev(m.seq_lens, torch.int32), m.scale, ws)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out), ref_o, f"mla B=600 S={S}")
        assert_lse_close(lse.cpu().numpy(), ref_l, f"mla B=600 lse S={S}")
    assert pa.pa_get_device_error() == 0
