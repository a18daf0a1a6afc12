"""Seeded random shapes through the whole standard-pool path, against the
oracle, every row: the cache write (bf16 and fp8, bit-exact), varlen
attention (causal, non-causal or with a sliding window), split-KV decode of
each request's last row and the LSE merge (bf16 and fp8 pools), at a random
split count.  Each case draws the kv-head count, the group size (1-16), the
head size (64 / 128), the block size (a multiple of 16, powers of two and
not), the request count, lengths mixed with block-boundary values, and the
query lengths; the parametrised tests elsewhere walk these axes one at a
time, this one crosses them.  Further sets do the same for MLA latent
decode (head count, block size, batch, lengths, split count), cascade
attention (prefix length, suffixes, decode or prefill rows, masking, both
split counts) and MLA prefill (head count, block size, lengths, masking),
and a last set takes larger batches (grids of thousands of CTAs) with the
varlen rows sampled.
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
    # fp8 scales, log-uniform over [0.002, 0.04]: at the small end many new
    # keys and values saturate at +-448 codes.  The pool's cached entries are
    # random codes (up to 448 * scale), so the upper end keeps them below ~18:
    # with values in the hundreds, an output that is a small difference of
    # large weighted terms is only as exact as the weights (f16, 2^-11), and
    # the absolute 1e-2 bar is meant for values of unit scale.
    ks, vs = (float(np.exp(rng.uniform(np.log(0.002), np.log(0.04)))) for _ in range(2))
    # Softmax scale, log-uniform over [1/4, 4] / sqrt(d): from flat rows to
    # rows dominated by a few tokens.
    scale = float(np.exp(rng.uniform(np.log(0.25), np.log(4.0)))) / np.sqrt(d)
    return dict(hkv=hkv, g=g, d=d, bs=bs, seq=seq, ql=ql, mode=mode, window=window, S=splits,
                ks=ks, vs=vs, scale=scale)


@pytest.mark.parametrize("seed", SEEDS)
def test_random_shape(pa, seed):
    c = draw_case(seed)
    hq = c["hkv"] * c["g"]
    b = workloads.make_paged_batch(f"fuzz{seed}", 4100 + seed, c["seq"], c["ql"], hq, c["hkv"],
                                   c["d"], c["bs"], causal=c["mode"] != "noncausal",
                                   scale=c["scale"])
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
    # The same batch over an fp8 pool at the case's scales: quantising write
    # (bit-exact), decode.
    p8 = workloads.fp8_pool(b)
    d8 = torch.from_numpy(p8.copy()).cuda()
    ks, vs = c["ks"], c["vs"]
    pa.pa_reshape_and_cache_fp8(to_dev_bf16(b.key), to_dev_bf16(b.value), d8,
                                to_dev(b.slot_mapping, torch.int64), ks, vs)
    ref8 = oracle.reshape_and_cache_fp8(b.key, b.value, p8, b.slot_mapping, c["bs"], ks, vs)
    assert np.array_equal(d8.cpu().numpy(), ref8), what
    r8o, r8l = oracle.lse_merge(oracle.split_partials_fp8(b.q[last], ref8, b.block_table,
                                                          b.seq_lens, b.scale, ks, vs, 1))
    ws = pa.decode_workspace(n, hq, c["S"], c["d"])
    out, lse = pa.pa_decode_fp8(q, d8, table, seql, b.scale, ks, vs, ws)
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
    scale = float(np.exp(rng.uniform(np.log(0.25), np.log(4.0)))) / np.sqrt(192.0)
    return dict(heads=heads, bs=bs, seq=seq, S=splits, scale=scale)


@pytest.mark.parametrize("seed", list(range(24)))
def test_random_mla_decode(pa, seed):
    c = draw_mla_case(seed)
    m = workloads.make_mla_batch(f"mla_fuzz{seed}", 5100 + seed, c["seq"], c["heads"],
                                 block_size=c["bs"], scale=c["scale"])
    ref_o, ref_l = oracle.mla_decode(m.q, m.pool, m.block_table, m.seq_lens, m.scale)
    ws = pa.decode_workspace(m.batch, c["heads"], c["S"], 512)
    out, lse = pa.pa_mla_decode(to_dev_bf16(m.q), to_dev_bf16(m.pool),
                                to_dev(m.block_table, torch.int32),
                                to_dev(m.seq_lens, torch.int32), m.scale, ws)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o, f"mla seed {seed} {c}")
    assert_lse_close(lse.cpu().numpy(), ref_l, f"mla lse seed {seed} {c}")
    assert pa.pa_get_device_error() == 0


def draw_cascade_case(seed):
    """Shape of cascade case `seed`: a shared prefix of 1-39 blocks, 1-6
    requests with their own suffixes, decode (one query each) or prefill
    rows, causal or not, and the two split counts."""
    rng = np.random.default_rng(6000 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    while hkv * g > 32:
        hkv //= 2
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32, 64]))
    prefix_blocks = int(rng.integers(1, 40))
    n = int(rng.integers(1, 7))
    decode = bool(rng.random() < 0.5)
    suf = [int(rng.integers(1, 400)) for _ in range(n)]
    ql = [1] * n if decode else [int(min(x, rng.integers(1, 150))) for x in suf]
    causal = True if decode else bool(rng.random() < 0.7)
    return dict(hkv=hkv, g=g, d=d, bs=bs, P=prefix_blocks, suf=suf, ql=ql, causal=causal,
                S1=int(rng.integers(1, 7)), S2=int(rng.integers(1, 5)))


@pytest.mark.parametrize("seed", list(range(24)))
def test_random_cascade(pa, seed):
    from tests.test_gpu_parity import Dev
    c = draw_cascade_case(seed)
    hq = c["hkv"] * c["g"]
    b = workloads.make_shared_prefix_batch(f"casc_fuzz{seed}", 6100 + seed, c["P"], c["suf"],
                                           c["ql"], hq, c["hkv"], c["d"], c["bs"])
    dev = Dev(pa, b)
    pool = dev.ref_pool()
    ref_o, ref_l = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc,
                                          b.seq_lens, b.scale, causal=c["causal"])
    ws = pa.cascade_workspace(b.num_tokens, hq, c["S1"], c["S2"], c["d"])
    out, lse = pa.pa_cascade_fwd(dev.q, dev.pool, dev.table, dev.qsl, dev.seq,
                                 int(b.query_lens.max()), c["P"], b.scale, ws, c["S1"],
                                 causal=c["causal"])
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o, f"cascade seed {seed} {c}")
    assert_lse_close(lse.cpu().numpy(), ref_l, f"cascade lse seed {seed} {c}")
    assert pa.pa_get_device_error() == 0


def draw_mla_prefill_case(seed):
    """Shape of MLA prefill case `seed`: head count, block size, 1-4
    requests, context and new-token lengths, causal or not."""
    rng = np.random.default_rng(7000 + seed)
    heads = int(rng.choice([4, 8, 16, 20, 32, 128]))
    bs = int(rng.choice([16, 32, 64, 128]))
    n = int(rng.integers(1, 5))
    top = 200 if heads == 128 else 400
    seq = [int(rng.integers(1, top)) for _ in range(n)]
    ql = [int(min(x, rng.integers(1, 200))) for x in seq]
    return dict(heads=heads, bs=bs, seq=seq, ql=ql, causal=bool(rng.random() < 0.8))


@pytest.mark.parametrize("seed", list(range(12)))
def test_random_mla_prefill(pa, seed):
    """The output within the usual tolerance of the oracle's.  The LSE
    within 1e-3 plus what the expansion's own rounding can move it by: the
    kernel accumulates each expanded key element in fp32 and rounds it to
    bf16, the oracle rounds the fp64 product, and where the sum lies that
    close to a rounding boundary the two pick neighbouring bf16 values (the
    expansion test bounds this by one unit in the last place).  A key that
    moves by dK moves a score by at most scale * sum_e |q_e| |dK_e|, and the
    LSE by at most the largest such score shift over the visible tokens; the
    allowance is that shift, from the kernel's expanded keys (read back from
    the workspace) against the oracle's."""
    from tests.test_gpu_mla_prefill import _expanded_ref, _written_pool
    c = draw_mla_prefill_case(seed)
    b = workloads.make_mla_prefill_batch(f"mlap_fuzz{seed}", 7100 + seed, c["seq"], c["ql"],
                                         c["heads"], block_size=c["bs"])
    pool = _written_pool(b)
    n_req, heads = b.num_seqs, b.num_heads
    s_max = int(b.seq_lens.max())
    # Zeroed so that the slots past each request's length (never written)
    # convert cleanly when the expanded keys are read back.
    ws = torch.zeros(pa.pa_mla_prefill_workspace_bytes(n_req, s_max, heads), dtype=torch.uint8,
                     device="cuda")
    out, lse = pa.pa_mla_prefill(to_dev_bf16(b.q), to_dev_bf16(pool), to_dev_bf16(b.w_kv_b),
                                 to_dev(b.block_table, torch.int32),
                                 to_dev(b.query_start_loc, torch.int32),
                                 to_dev(b.seq_lens, torch.int32), int(b.query_lens.max()),
                                 b.scale, ws, causal=c["causal"])
    torch.cuda.synchronize()
    what = f"mla prefill seed {seed} {c}"
    ref_o, ref_l = oracle.mla_prefill(b.q, pool, b.w_kv_b, b.block_table, b.query_start_loc,
                                      b.seq_lens, b.scale, causal=c["causal"])
    assert_out_close(bf16_to_f64(out), ref_o, what)
    got_l = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got_l), np.isneginf(ref_l)), what
    k_gpu = bf16_to_f64(ws[: n_req * s_max * heads * 192 * 2].view(torch.bfloat16)
                        .view(n_req, s_max, heads, 192))
    q_abs = np.abs(workloads.bf16_bits_to_f32(b.q).astype(np.float64))
    qsl = b.query_start_loc
    for i in range(n_req):
        rows = slice(int(qsl[i]), int(qsl[i + 1]))
        n, ql = int(b.seq_lens[i]), int(qsl[i + 1] - qsl[i])
        if ql == 0:
            continue
        k_ref, _, _ = _expanded_ref(b, pool, i, np.arange(heads))
        dk = np.abs(k_gpu[i, :n] - k_ref)                                     # [n, h, 192]
        shift = b.scale * np.einsum("rhe,phe->rhp", q_abs[rows], dk)          # [ql, h, n]
        if c["causal"]:
            pos = n - ql + np.arange(ql)
            shift = np.where(np.arange(n)[None, None, :] <= pos[:, None, None], shift, 0.0)
        allow = 1e-3 + shift.max(axis=2)
        err = np.abs(got_l[rows] - ref_l[rows])
        fin = np.isfinite(ref_l[rows])
        bad = fin & (err > allow)
        assert not bad.any(), (f"{what}: request {i}: LSE error {err[fin].max():.3e} beyond "
                               f"1e-3 + the expansion's rounding shift")
    assert pa.pa_get_device_error() == 0


def draw_large_case(seed):
    """A larger random batch: up to 64 requests of up to 8192 tokens, either
    prefill-like (up to 2048 new rows each) or decode-like (up to 8), any
    masking, up to 64 splits; grids of thousands of CTAs."""
    rng = np.random.default_rng(9000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32, 64, 128]))
    n = int(rng.integers(1, 65))
    seq = rng.integers(1, 8193, size=n)
    top = 2049 if rng.random() < 0.5 else 9
    ql = np.minimum(seq, rng.integers(1, top, size=n))
    causal = bool(rng.random() < 0.8)
    return dict(hkv=hkv, g=g, d=d, bs=bs, seq=seq, ql=ql, causal=causal,
                S=int(rng.integers(1, 65)), rng=rng)


@pytest.mark.parametrize("seed", list(range(10)))
def test_random_large_shape(pa, seed):
    """Varlen attention on every request's first and last row and 300 random
    rows, and split-KV decode of every request's last row, against the
    oracle."""
    c = draw_large_case(seed)
    rng = c.pop("rng")
    hq = c["hkv"] * c["g"]
    b = workloads.make_paged_batch(f"large{seed}", 9100 + seed, c["seq"], c["ql"], hq, c["hkv"],
                                   c["d"], c["bs"], causal=c["causal"])
    what = f"seed {seed} hkv {c['hkv']} g {c['g']} d {c['d']} bs {c['bs']} n {len(c['seq'])} " \
           f"T {b.num_tokens} causal {c['causal']} S {c['S']}"
    pool = to_dev_bf16(b.pool)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key), to_dev_bf16(b.value), pool,
                            to_dev(b.slot_mapping, torch.int64))
    ref_pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, c["bs"])
    assert np.array_equal(bf16_bits(pool), ref_pool), what
    table, seql = to_dev(b.block_table, torch.int32), to_dev(b.seq_lens, torch.int32)
    qsl = b.query_start_loc
    out, lse = pa.pa_varlen_fwd(to_dev_bf16(b.q), pool, table, to_dev(qsl, torch.int32), seql,
                                int(b.query_lens.max()), b.scale, causal=c["causal"])
    torch.cuda.synchronize()
    mask = np.zeros(b.num_tokens, np.uint8)
    mask[qsl[:-1]] = 1
    mask[qsl[1:] - 1] = 1
    mask[rng.choice(b.num_tokens, size=min(b.num_tokens, 300), replace=False)] = 1
    ref_o, ref_l = oracle.paged_attention(b.q, ref_pool, b.block_table, qsl, b.seq_lens, b.scale,
                                          causal=c["causal"], row_mask=mask)
    sel = mask.astype(bool)
    assert_out_close(bf16_to_f64(out)[sel], ref_o[sel], f"varlen {what}")
    assert_lse_close(lse.cpu().numpy()[sel], ref_l[sel], f"varlen lse {what}")
    last = qsl[1:] - 1
    n = b.num_seqs
    q = to_dev_bf16(b.q[last]).view(n, hq, c["d"])
    ref_o, ref_l = oracle.lse_merge(
        oracle.split_partials(b.q[last], ref_pool, b.block_table, b.seq_lens, b.scale, 1))
    ws = pa.decode_workspace(n, hq, c["S"], c["d"])
    out, lse = pa.pa_decode(q, pool, table, seql, b.scale, ws)
    torch.cuda.synchronize()
    assert_out_close(bf16_to_f64(out), ref_o, f"decode {what}")
    assert_lse_close(lse.cpu().numpy(), ref_l, f"decode lse {what}")
    assert pa.pa_get_device_error() == 0
