"""Block sizes that are multiples of 16 but not powers of two (48, 80), and a
large one (256), through the cache writes, varlen attention, split-KV decode
(bf16 and fp8) and MLA decode (96: a multiple of 32), against the oracle.
The fp8 kernel splits a token index into (block, offset) with a shift and a
mask when the block size is a power of two and by division otherwise; both
paths run here.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import (assert_lse_close, assert_out_close, bf16_bits, bf16_to_f64, to_dev,
                          to_dev_bf16)

pytestmark = pytest.mark.gpu

KS, VS = workloads.FP8_K_SCALE, workloads.FP8_V_SCALE


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


@pytest.mark.parametrize("bs", [48, 80, 256])
def test_standard_pool_block_sizes(pa, bs):
    seq, ql = [1, 47, 48, 49, 300, 1000], [1, 20, 1, 49, 130, 3]
    b = workloads.make_paged_batch(f"bs{bs}", 100 + bs, seq, ql, 16, 4, 128, bs)
    pool = to_dev_bf16(b.pool)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key), to_dev_bf16(b.value), pool,
                            to_dev(b.slot_mapping, torch.int64))
    ref_pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, bs)
    assert np.array_equal(bf16_bits(pool), ref_pool)
    table, seql = to_dev(b.block_table, torch.int32), to_dev(b.seq_lens, torch.int32)
    ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    out, lse = pa.pa_varlen_fwd(to_dev_bf16(b.q), pool, table, to_dev(b.query_start_loc, torch.int32),
                                seql, int(b.query_lens.max()), b.scale)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o, f"varlen bs={bs}")
    assert_lse_close(lse.cpu().numpy(), ref_l, f"varlen lse bs={bs}")
    last = b.query_start_loc[1:] - 1
    N = b.num_seqs
    q = to_dev_bf16(b.q[last]).view(N, 16, 128)
    for S in (1, 3):
        ws = pa.decode_workspace(N, 16, S, 128)
        out, lse = pa.pa_decode(q, pool, table, seql, b.scale, ws)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out), ref_o[last], f"decode bs={bs} S={S}")
        assert_lse_close(lse.cpu().numpy(), ref_l[last], f"decode lse bs={bs} S={S}")
    # The same batch over an fp8 pool.
    p8 = workloads.fp8_pool(b)
    d8 = torch.from_numpy(p8.copy()).cuda()
    pa.pa_reshape_and_cache_fp8(to_dev_bf16(b.key), to_dev_bf16(b.value), d8,
                                to_dev(b.slot_mapping, torch.int64), KS, VS)
    ref8 = oracle.reshape_and_cache_fp8(b.key, b.value, p8, b.slot_mapping, bs, KS, VS)
    assert np.array_equal(d8.cpu().numpy(), ref8)
    r8o, r8l = oracle.lse_merge(oracle.split_partials_fp8(b.q[last], ref8, b.block_table,
                                                          b.seq_lens, b.scale, KS, VS, 1))
    for S in (1, 3):
        ws = pa.decode_workspace(N, 16, S, 128)
        out, lse = pa.pa_decode_fp8(q, d8, table, seql, b.scale, KS, VS, ws)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out), r8o, f"fp8 decode bs={bs} S={S}")
        assert_lse_close(lse.cpu().numpy(), r8l, f"fp8 decode lse bs={bs} S={S}")
    assert pa.pa_get_device_error() == 0


def test_mla_block_size_96(pa):
    m = workloads.make_mla_batch("mla_bs96", 109, [1, 95, 96, 97, 700, 0], 128, block_size=96,
                                 scale=1.0 / math.sqrt(192.0))
    ref_o, ref_l = oracle.mla_decode(m.q, m.pool, m.block_table, m.seq_lens, m.scale)
    for S in (1, 2):
        ws = pa.decode_workspace(m.batch, 128, S, 512)
        out, lse = pa.pa_mla_decode(to_dev_bf16(m.q), to_dev_bf16(m.pool),
                                    to_dev(m.block_table, torch.int32),
                                    to_dev(m.seq_lens, torch.int32), m.scale, ws)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out), ref_o, f"mla bs=96 S={S}")
        assert_lse_close(lse.cpu().numpy(), ref_l, f"mla lse bs=96 S={S}")
    assert pa.pa_get_device_error() == 0
