"""Varlen attention and split-KV decode at large logits, against the oracle.

With N(0, 1) inputs every softmax row spreads its weight over many tokens
and the bf16 rounding of the weights averages out.  With queries scaled by 4
or 8 (scaled logits of tens), a few tokens dominate each row; the kernels'
outputs must then still be weighted means of the value rows, i.e. the
divisor must be the sum of the very (bf16-rounded) weights that the PV
product multiplies, while the LSE uses the unrounded ones.  All rows / all
requests, all heads.
"""

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


def _scaled(b, factor):
    q = workloads.bf16_bits_to_f32(b.q) * np.float32(factor)   # a power of two: exact
    b.q = workloads.f32_to_bf16_bits(q)
    return b


def _written_pool(pa, b):
    pool = to_dev_bf16(b.pool)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key), to_dev_bf16(b.value), pool,
                            to_dev(b.slot_mapping, torch.int64))
    ref = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    return pool, ref


CASES = {
    # name: (seed, seq_lens, query_lens, Hq, Hkv, d, bs)
    "d128_g4": (81, [700, 130, 2100, 64], [260, 130, 300, 17], 32, 8, 128, 16),
    "d64_g2_bs32": (82, [300, 97, 1500], [120, 3, 200], 8, 4, 64, 32),
}


@pytest.mark.parametrize("factor", [4, 8])
@pytest.mark.parametrize("name", sorted(CASES))
def test_varlen_large_logits_all_rows(pa, name, factor):
    seed, seq, ql, hq, hkv, hd, bs = CASES[name]
    b = _scaled(workloads.make_paged_batch(name, seed, seq, ql, hq, hkv, hd, bs), factor)
    pool, ref_pool = _written_pool(pa, b)
    out, lse = pa.pa_varlen_fwd(to_dev_bf16(b.q), pool, to_dev(b.block_table, torch.int32),
                                to_dev(b.query_start_loc, torch.int32),
                                to_dev(b.seq_lens, torch.int32), int(b.query_lens.max()), b.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    assert np.abs(ref_l).max() > 8.0 * factor / 4     # the rows are peaked
    assert_out_close(bf16_to_f64(out), ref_o, f"varlen {name} x{factor}")
    assert_lse_close(lse.cpu().numpy(), ref_l, f"varlen {name} x{factor} lse")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("factor", [4, 8])
@pytest.mark.parametrize("hq,hkv,hd", [(32, 8, 128), (16, 1, 128), (8, 2, 64)])
def test_decode_large_logits_all_requests(pa, hq, hkv, hd, factor):
    seq = [1, 17, 300, 1024, 4096, 2500]
    b = _scaled(workloads.make_paged_batch(f"dec{hq}_{hd}", 83, seq, [1] * len(seq), hq, hkv,
                                           hd, 16), factor)
    pool, ref_pool = _written_pool(pa, b)
    ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale)
    N = b.num_seqs
    q = to_dev_bf16(b.q).view(N, hq, hd)
    table, seql = to_dev(b.block_table, torch.int32), to_dev(b.seq_lens, torch.int32)
    for S in (1, 5):
        ws = pa.decode_workspace(N, hq, S, hd)
        out, lse = pa.pa_decode(q, pool, table, seql, b.scale, ws)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out), ref_o, f"decode x{factor} S={S}")
        assert_lse_close(lse.cpu().numpy(), ref_l, f"decode x{factor} S={S} lse")
    assert pa.pa_get_device_error() == 0
