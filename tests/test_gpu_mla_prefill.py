"""GPU parity of the MLA prefill (multi-head formulation) through the C ABI
against the fp64 oracle.

Step 1, the expansion of each context token's latent through kv_b_proj, is
checked value by value: the expanded key and value parts may differ from the
oracle's bf16-rounded fp64 products by one bf16 unit in the last place (the
GPU accumulates in fp32, so a sum within fp32 rounding of a bf16 rounding
boundary may round the other way), the copied k_pe part is bit-exact.  Step 2
(attention over the expanded keys and values) and the whole call are checked
against the oracle's mla_prefill with the tolerances of ``tests/parity.py``.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import (BF16_NAN, assert_lse_close, assert_out_close, bf16_bits, bf16_to_f64,
                          bf16_ulp, to_dev, to_dev_bf16)

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


def _f64(bits):
    return workloads.bf16_bits_to_f32(bits).astype(np.float64)


def _written_pool(b, poison=True):
    pool = oracle.mla_cache_write(b.kv_c, b.k_pe, b.pool, b.slot_mapping, b.block_size)
    if poison:
        used = np.zeros((b.num_blocks, b.block_size), bool)
        for i in range(b.num_seqs):
            pos = np.arange(int(b.seq_lens[i]))
            used[b.block_table[i, pos // b.block_size], pos % b.block_size] = True
        pool[~used] = BF16_NAN
    return pool


def _expanded_ref(b, pool, i, heads):
    """Oracle-side expansion of request i for the given heads: (K [n, h, 192],
    V [n, h, 128]) as float64, the products rounded to bf16, and the sums of
    |w c| terms of each product [n, h, 256] (for the fp32 error bound)."""
    n = int(b.seq_lens[i])
    pos = np.arange(n)
    rows = _f64(pool[b.block_table[i, pos // b.block_size], pos % b.block_size])   # [n, 576]
    W = _f64(b.w_kv_b[heads])                                                        # [h, 256, 512]
    kv = oracle.round_bf16(np.einsum("hor,nr->nho", W, rows[:, :512]))               # [n, h, 256]
    mag = np.einsum("hor,nr->nho", np.abs(W), np.abs(rows[:, :512]))
    K = np.concatenate([kv[:, :, :128], np.broadcast_to(rows[:, None, 512:],
                                                        (n, len(heads), 64))], axis=2)
    return K, kv[:, :, 128:], mag


def _assert_close_to_rounded(got, ref, mag, what):
    """|got - ref| <= one bf16 ulp of ref + 2 * 512 * 2^-24 * sum |w c|: the
    rounding of the result plus twice the worst-case error of a 512-term fp32
    accumulation (which dominates near zero, where terms cancel)."""
    err = np.abs(got - ref)
    bad = err > bf16_ulp(ref) + 2.0 ** -14 * mag
    assert not bad.any(), f"{what}: {int(bad.sum())} values beyond the bound"


@pytest.mark.parametrize("heads,bs", [(16, 64), (20, 16), (128, 128)])
def test_mla_expand_matches_oracle(pa, heads, bs):
    seq = [1, 127, 128, 129, 300]
    b = workloads.make_mla_prefill_batch(f"mla_exp_{heads}_{bs}", 91, seq, [1] * len(seq), heads,
                                         block_size=bs)
    pool = _written_pool(b)
    S = int(b.seq_lens.max())
    k_ws, v_ws = pa.mla_prefill_workspace(b.num_seqs, S, heads)
    k_ws.zero_()   # rows past each sequence are not written; keep them finite for the copy
    v_ws.zero_()
    pa.pa_mla_expand_kv(to_dev_bf16(pool), to_dev_bf16(b.w_kv_b), to_dev(b.block_table, torch.int32),
                        to_dev(b.seq_lens, torch.int32), k_ws, v_ws)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    K, V = bf16_to_f64(k_ws), bf16_to_f64(v_ws)
    sel = list(range(heads)) if heads <= 20 else [0, 1, 63, 64, 127]
    for i in range(b.num_seqs):
        n = int(b.seq_lens[i])
        rk, rv, mag = _expanded_ref(b, pool, i, sel)
        _assert_close_to_rounded(K[i, :n][:, sel, :128], rk[:, :, :128], mag[:, :, :128],
                                 f"k_nope req {i}")
        assert np.array_equal(K[i, :n][:, sel, 128:], rk[:, :, 128:]), f"k_pe req {i}"
        _assert_close_to_rounded(V[i, :n][:, sel], rv, mag[:, :, 128:], f"v req {i}")
        # Most values are bit-identical to the oracle's rounding.
        assert np.mean(K[i, :n][:, sel, :128] == rk[:, :, :128]) > 0.99


def _prefill(pa, b, pool, causal=True):
    d_pool = to_dev_bf16(pool)
    S = int(b.seq_lens.max())
    ws = torch.empty(pa.pa_mla_prefill_workspace_bytes(b.num_seqs, S, b.num_heads),
                     dtype=torch.uint8, device="cuda")
    out, lse = pa.pa_mla_prefill(to_dev_bf16(b.q), d_pool, to_dev_bf16(b.w_kv_b),
                                 to_dev(b.block_table, torch.int32),
                                 to_dev(b.query_start_loc, torch.int32),
                                 to_dev(b.seq_lens, torch.int32), int(b.query_lens.max()),
                                 b.scale, ws, causal=causal)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


MLA_PREFILL_CASES = {
    # name: (seed, seq_lens, query_lens, heads, block_size)
    "ragged_h16_bs64": (92, [1, 70, 200, 129, 64], [1, 70, 130, 1, 17], 16, 64),
    "h4_bs16_long_rows": (93, [300, 45], [260, 45], 4, 16),
    "h128_bs128": (94, [150, 33], [100, 33], 128, 128),
}


@pytest.mark.parametrize("name", sorted(MLA_PREFILL_CASES))
def test_mla_prefill_all_rows(pa, name):
    seed, seq, ql, heads, bs = MLA_PREFILL_CASES[name]
    b = workloads.make_mla_prefill_batch(name, seed, seq, ql, heads, block_size=bs)
    pool = _written_pool(b)
    out, lse = _prefill(pa, b, pool)
    ref_o, ref_l = oracle.mla_prefill(b.q, pool, b.w_kv_b, b.block_table, b.query_start_loc,
                                      b.seq_lens, b.scale)
    assert_out_close(out, ref_o, f"{name} out")
    assert_lse_close(lse, ref_l, f"{name} lse")
    assert pa.pa_get_device_error() == 0


def test_mla_prefill_non_causal(pa):
    seed, seq, ql, heads, bs = MLA_PREFILL_CASES["ragged_h16_bs64"]
    b = workloads.make_mla_prefill_batch("nc", seed, seq, ql, heads, block_size=bs)
    pool = _written_pool(b)
    out, lse = _prefill(pa, b, pool, causal=False)
    ref_o, ref_l = oracle.mla_prefill(b.q, pool, b.w_kv_b, b.block_table, b.query_start_loc,
                                      b.seq_lens, b.scale, causal=False)
    assert_out_close(out, ref_o, "non-causal out")
    assert_lse_close(lse, ref_l, "non-causal lse")


def test_mla_prefill_workload_full_size_sampled(pa):
    b = workloads.mla_prefill()
    pool = _written_pool(b, poison=False)
    out, lse = _prefill(pa, b, pool)
    # Every Q tile's first and last row (the MLA attention has one q head per
    # kv head, so a 128-row tile is 128 query rows) plus 1 % random rows, in
    # 8 heads spread over the 128.
    rng = np.random.default_rng(97)
    rows = np.zeros(b.num_tokens, np.uint8)
    for i in range(b.num_seqs):
        a, e = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
        starts = np.arange(a, e, 128)
        rows[starts] = 1
        rows[np.minimum(starts + 127, e - 1)] = 1
    rows[rng.choice(b.num_tokens, b.num_tokens // 100, replace=False)] = 1
    heads = np.zeros(b.num_heads, np.uint8)
    heads[[0, 17, 38, 64, 77, 101, 126, 127]] = 1
    ref_o, ref_l = oracle.mla_prefill(b.q, pool, b.w_kv_b, b.block_table, b.query_start_loc,
                                      b.seq_lens, b.scale, head_mask=heads, row_mask=rows)
    r, h = rows.astype(bool), heads.astype(bool)
    assert_out_close(out[r][:, h], ref_o[r][:, h], "mla prefill out")
    assert_lse_close(lse[r][:, h], ref_l[r][:, h], "mla prefill lse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert pa.pa_get_device_error() == 0
