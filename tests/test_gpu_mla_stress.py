"""MLA latent decode at large logits, all heads, against the fp64 oracle.

The MLA kernel splits each 576-wide score over a CTA pair and sends one
CTA's partial scores to the other as 16-bit fixed point, in units of the
row's largest partial / 32767; the error of a score is then at most
max |partial| / 65534 of that row and tile.  The small-logit cases of
test_gpu_parity.py do not reach that bound.  These batches do:

* queries scaled so the scaled logits reach about +-45 and +-90;
* one planted outlier token per request, ~20 above every other logit of
  every head (all heads share a query component that the outlier row
  points along);
* heads whose partial scores differ by 2^10 inside one tile (half the heads
  scaled by 4, the other half by 2^-8).

Each runs with one split (the kernel writes the output) and three (the
partials go through the LSE merge).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import assert_lse_close, assert_out_close, bf16_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

SEQ = [1, 63, 64, 65, 700, 2000, 4096, 0]
SCALE = 1.0 / math.sqrt(192.0)


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


def _f32(bits):
    return workloads.bf16_bits_to_f32(bits)


def _bits(x):
    return workloads.f32_to_bf16_bits(np.asarray(x, np.float32))


def _batch(kind):
    """(batch, outlier targets): targets[i] is the logit the planted row of
    request i was aimed at (outlier batches only)."""
    b = workloads.make_mla_batch(f"mla_stress_{kind}", 61, SEQ, 128, scale=SCALE)
    targets = {}
    q = _f32(b.q)
    if kind == "logits45":
        b.q = _bits(q * 6.0)
    elif kind == "logits90":
        b.q = _bits(q * 10.0)
    elif kind == "head_ratio":
        f = np.where(np.arange(128) < 64, 4.0, 2.0 ** -8).astype(np.float32)
        b.q = _bits(q * f[None, :, None])
    elif kind == "outlier":
        rng = np.random.default_rng(62)
        u = rng.standard_normal((b.batch, 576)).astype(np.float32)
        b.q = _bits(q + u[:, None, :])
        qf = _f32(b.q).astype(np.float64)
        pool = b.pool.copy()
        for i, n in enumerate(b.seq_lens):
            if n == 0:
                continue
            p = int(rng.integers(0, n))
            blk = int(b.block_table[i, p // b.block_size])
            ctx = pool[b.block_table[i, :(n + b.block_size - 1) // b.block_size]].reshape(
                -1, 576)[:n]
            rest = SCALE * (qf[i] @ _f32(ctx).astype(np.float64).T)        # [H, n]
            # The outlier row k = kappa u makes every head's logit about
            # kappa * SCALE * |u|^2; kappa puts it 20 above the batch row's max.
            targets[i] = rest.max() + 20.0
            kappa = targets[i] / (SCALE * float(u[i] @ u[i]))
            pool[blk, p % b.block_size] = _bits(kappa * u[i])
        b.pool = pool
    else:
        raise ValueError(kind)
    return b, targets


def _run(pa, b, S):
    ws = pa.decode_workspace(b.batch, b.num_heads, S, b.kv_lora_rank)
    out, lse = pa.pa_mla_decode(to_dev_bf16(b.q), to_dev_bf16(b.pool),
                                to_dev(b.block_table, torch.int32),
                                to_dev(b.seq_lens, torch.int32), b.scale, ws)
    torch.cuda.synchronize()
    return bf16_to_f64(out), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("kind", ["logits45", "logits90", "outlier", "head_ratio"])
def test_mla_large_logits_all_heads(pa, kind):
    b, targets = _batch(kind)
    ref_o, ref_l = oracle.mla_decode(b.q, b.pool, b.block_table, b.seq_lens, b.scale)
    fin = np.isfinite(ref_l)
    top = float(np.abs(ref_l[fin]).max())
    if kind == "logits45":
        assert top > 35.0, top          # the batch reaches the range it names
    if kind == "logits90":
        assert top > 70.0, top
    if kind == "outlier":
        # The planted row dominates every head: each head's LSE is close to
        # the aimed logit (the heads' own query parts move it by ~10 %),
        # far above the other rows' best.
        for i, tgt in targets.items():
            assert np.all(ref_l[i] > 0.75 * tgt) and np.all(ref_l[i] < 1.25 * tgt), (i, tgt)
    for S in (1, 3):
        out, lse = _run(pa, b, S)
        assert_out_close(out, ref_o, f"mla {kind} S={S}")
        assert_lse_close(lse, ref_l, f"mla {kind} lse S={S}")
    assert pa.pa_get_device_error() == 0
