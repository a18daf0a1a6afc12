"""Seeded random shapes through the whole standard-pool path, against the
oracle, every row: the cache write (bf16 and fp8, bit-exact), varlen
attention (causal, non-causal or with a sliding window), split-KV decode of
each request's last row and the LSE merge (bf16 and fp8 pools), at a random
split count.  Each case draws the kv-head count, the group size (1-16), the
head size (64 / 128), the block size (a multiple of 16, powers of two and
not), the request count, lengths mixed with block-boundary values, and the
query lengths; the parametrised tests elsewhere walk these axes one at a
time, this one crosses them.  A second set does the same for MLA latent
decode (head count, block size, batch, lengths, split count).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import (assert_lse_close, assert_out_close, bf16_bits, bf16_to_f64, to_dev,
                          to_dev_bf16)

pytestmark = pytest.mark.gpu

KS, VS = workloads.FP8_K_SCALE, workloads.FP8_V_SCALE
SEEDS = list(range(64))


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


def draw_case(seed):
    """The shape of case `seed` (a plain function of the seed)."""
    rng = np.random.default_rng(4000 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    while hkv * g > 32:
        hkv //= 2
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32, 48, 64, 80, 128]))
    n = int(rng.integers(1, 7))
    edges = [1, bs - 1, bs, bs + 1, 127, 128, 129, 2 * bs]
    seq = [int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 1200))
           for _ in range(n)]
    seq = [max(1, x) for x in seq]
    ql = [int(min(x, rng.integers(1, 200))) for x in seq]
    mode = str(rng.choice(["causal", "noncausal", "window"]))
    window = int(rng.integers(1, 600))
    splits = int(rng.integers(1, 9))
    return dict(hkv=hkv, g=g, d=d, bs=bs, seq=seq, ql=ql, mode=mode, window=window, S=splits)


@pytest.mark.parametrize("seed", SEEDS)
def test_random_shape(pa, seed):
    c = draw_case(seed)
    hq = c["hkv"] * c["g"]
    b = workloads.make_paged_batch(f"fuzz{seed}", 4100 + seed, c["seq"], c["ql"], hq, c["hkv"],
                                   c["d"], c["bs"], causal=c["mode"] != "noncausal")
    what = f"seed {seed} {c}"
    # Cache write, bit-exact.
    pool = to_dev_bf16(b.pool)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key), to_dev_bf16(b.value), pool,
                            to_dev(b.slot_mapping, torch.int64))
    ref_pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, c["bs"])
    assert np.array_equal(bf16_bits(pool), ref_pool), what
    table, seql = to_dev(b.block_table, torch.int32), to_dev(b.seq_lens, torch.int32)
    qsl = to_dev(b.query_start_loc, torch.int32)
    mq = int(b.query_lens.max())
    # Varlen attention, every row.
    if c["mode"] == "window":
        out, lse = pa.pa_varlen_fwd_window(to_dev_bf16(b.q), pool, table, qsl, seql, mq, b.scale,
                                           c["window"])
        ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                              b.seq_lens, b.scale, window=c["window"])
    else:
        causal = c["mode"] == "causal"
        out, lse = pa.pa_varlen_fwd(to_dev_bf16(b.q), pool, table, qsl, seql, mq, b.scale,
                                    causal=causal)
        ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                              b.seq_lens, b.scale, causal=causal)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o, f"varlen {what}")
    assert_lse_close(lse.cpu().numpy(), ref_l, f"varlen lse {what}")
    # Split-KV decode of each request's last row (the row that sees the
    # whole sequence), then the merge.
    last = b.query_start_loc[1:] - 1
    n = b.num_seqs
    q = to_dev_bf16(b.q[last]).view(n, hq, c["d"])
    ref_ld, ref_ll = oracle.lse_merge(
        oracle.split_partials(b.q[last], ref_pool, b.block_table, b.seq_lens, b.scale, 1))
    ws = pa.decode_workspace(n, hq, c["S"], c["d"])
    out, lse = pa.pa_decode(q, pool, table, seql, b.scale, ws)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_ld, f"decode {what}")
    assert_lse_close(lse.cpu().numpy(), ref_ll, f"decode lse {what}")
    # The same batch over an fp8 pool: quantising write (bit-exact), decode.
    p8 = workloads.fp8_pool(b)
    d8 = torch.from_numpy(p8.copy()).cuda()
    pa.pa_reshape_and_cache_fp8(to_dev_bf16(b.key), to_dev_bf16(b.value), d8,
                                to_dev(b.slot_mapping, torch.int64), KS, VS)
    ref8 = oracle.reshape_and_cache_fp8(b.key, b.value, p8, b.slot_mapping, c["bs"], KS, VS)
    assert np.array_equal(d8.cpu().numpy(), ref8), what
    r8o, r8l = oracle.lse_merge(oracle.split_partials_fp8(b.q[last], ref8, b.block_table,
                                                          b.seq_lens, b.scale, KS, VS, 1))
    ws = pa.decode_workspace(n, hq, c["S"], c["d"])
    out, lse = pa.pa_decode_fp8(q, d8, table, seql, b.scale, KS, VS, ws)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), r8o, f"fp8 decode {what}")
    assert_lse_close(lse.cpu().numpy(), r8l, f"fp8 decode lse {what}")
    assert pa.pa_get_device_error() == 0


def draw_mla_case(seed):
    """The shape of MLA case `seed`: head count, block size (a multiple of
    32), batch, lengths (0 allowed, tile and block boundaries mixed in) and
    split count."""
    rng = np.random.default_rng(5000 + seed)
    heads = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([32, 64, 96, 128]))
    batch = int(rng.integers(1, 10))
    edges = [0, 1, 63, 64, 65, bs - 1, bs, bs + 1, 2 * bs]
    seq = [int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 2500))
           for _ in range(batch)]
    if max(seq) == 0:
        seq[0] = 1   # a pool needs at least one block
    splits = int(rng.integers(1, 4))
    return dict(heads=heads, bs=bs, seq=seq, S=splits)


@pytest.mark.parametrize("seed", list(range(24)))
def test_random_mla_decode(pa, seed):
    import math
    c = draw_mla_case(seed)
    m = workloads.make_mla_batch(f"mla_fuzz{seed}", 5100 + seed, c["seq"], c["heads"],
                                 block_size=c["bs"], scale=1.0 / math.sqrt(192.0))
    ref_o, ref_l = oracle.mla_decode(m.q, m.pool, m.block_table, m.seq_lens, m.scale)
    ws = pa.decode_workspace(m.batch, c["heads"], c["S"], 512)
    out, lse = pa.pa_mla_decode(to_dev_bf16(m.q), to_dev_bf16(m.pool),
                                to_dev(m.block_table, torch.int32),
                                to_dev(m.seq_lens, torch.int32), m.scale, ws)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o, f"mla seed {seed} {c}")
    assert_lse_close(lse.cpu().numpy(), ref_l, f"mla lse seed {seed} {c}")
    assert pa.pa_get_device_error() == 0
