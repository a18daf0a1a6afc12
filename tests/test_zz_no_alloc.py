"""pa_decode_noalloc: split-KV decode for callers that cannot allocate device
memory (a host application that owns all device allocations and gives the
library no allocator, or a path that must never call cudaMalloc), so they
cannot hand the library a workspace.  The entry point keeps its split
partials in a fixed device array inside the library instead.

Checked here through the C ABI against the regular two-call path
(pa_decode_splitkv into a caller workspace + pa_lse_merge) and against the
fp64 oracle, within the parity tolerances, on two calls in a row with
different inputs (the shared array keeps the previous call's contents, which
must not leak into the next result), at head sizes 128 and 64, with and
without the LSE output, and with split counts that take either merge
kernel.  This file is collected last on purpose.
"""

import ctypes

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
    return pa


def _batch(seed, seq, hq=32, hkv=8, d=128):
    b = workloads.make_paged_batch(f"noalloc{seed}", seed, seq, [1] * len(seq), hq, hkv, d, 16)
    N = b.num_seqs
    return dict(
        b=b,
        q=to_dev_bf16(b.q).view(N, hq, d),
        pool=to_dev_bf16(b.pool),
        table=to_dev(b.block_table, torch.int32),
        seq=to_dev(b.seq_lens, torch.int32),
    )


def _regular(pa, d, S):
    b = d["b"]
    ws = pa.decode_workspace(b.num_seqs, b.num_q_heads, S, b.head_size)
    out, lse = pa.pa_decode(d["q"], d["pool"], d["table"], d["seq"], b.scale, ws)
    return out, lse


def _noalloc_cabi(pa, d, S, with_lse=True):
    """Direct C-ABI call of pa_decode_noalloc with raw device pointers
    (lse = NULL when with_lse is False)."""
    b = d["b"]
    N, hq, hd = b.num_seqs, b.num_q_heads, b.head_size
    out = torch.empty((N, hq, hd), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((N, hq), dtype=torch.float32, device="cuda") if with_lse else None
    shape = pa.PaShape(N, hq, b.num_kv_heads, hd, 16, b.num_blocks, b.max_blocks_per_seq)
    rc = pa.lib().pa_decode_noalloc(
        d["q"].data_ptr(), d["pool"].data_ptr(), d["table"].data_ptr(), d["seq"].data_ptr(),
        ctypes.byref(shape), ctypes.c_float(b.scale), S, int(b.seq_lens.max()), out.data_ptr(),
        lse.data_ptr() if with_lse else None, torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_OK, pa.status_string(rc)
    return out, lse


def _oracle(b):
    return oracle.paged_attention(b.q, b.pool, b.block_table, b.query_start_loc, b.seq_lens,
                                  b.scale)


def test_noalloc_matches_workspace_path_twice(pa):
    first = _batch(61, [3000, 17, 640, 1, 2049, 128])
    second = _batch(62, [95, 4096, 33, 700])
    for d, S in ((first, 8), (second, 5)):
        out_n, lse_n = _noalloc_cabi(pa, d, S)
        out_r, lse_r = _regular(pa, d, S)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out_n), bf16_to_f64(out_r), "noalloc vs workspace path")
        assert_lse_close(lse_n.cpu().numpy(), lse_r.cpu().numpy(), "noalloc lse")
        # And both against the oracle.
        ref_o, ref_l = _oracle(d["b"])
        assert_out_close(bf16_to_f64(out_n), ref_o, "noalloc vs oracle")
        assert_lse_close(lse_n.cpu().numpy(), ref_l, "noalloc lse vs oracle")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("hq,hkv,hd,S", [(8, 2, 64, 5), (32, 8, 128, 24)],
                         ids=["d64_warp_merge", "d128_S24_block_merge"])
def test_noalloc_other_shapes_without_lse(pa, hq, hkv, hd, S):
    """Head size 64, and 24 splits at head size 128 (more than the warp-wide
    merge takes, so the merge runs its shared-memory kernel), with lse = NULL;
    two calls in a row, each against the workspace path and the oracle."""
    for seed, seq in ((63, [1500, 3, 260, 4096, 17]), (64, [33, 1200, 640])):
        d = _batch(seed, seq, hq, hkv, hd)
        out_n, _ = _noalloc_cabi(pa, d, S, with_lse=False)
        out_r, _ = _regular(pa, d, S)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out_n), bf16_to_f64(out_r), f"noalloc d={hd} S={S}")
        ref_o, _ = _oracle(d["b"])
        assert_out_close(bf16_to_f64(out_n), ref_o, f"noalloc d={hd} S={S} vs oracle")
    assert pa.pa_get_device_error() == 0


def test_noalloc_rejects_sizes_beyond_the_array(pa):
    limit = pa.PA_NOALLOC_WORKSPACE_BYTES
    N, hq, d = 64, 32, 128
    S = limit // (N * hq * (d + 1) * 4) + 1       # one split too many
    shape = pa.PaShape(N, hq, 8, d, 16, 100, 10)
    rc = pa.lib().pa_decode_noalloc(16, 16, 16, 16, ctypes.byref(shape), ctypes.c_float(0.1), S,
                                    4096, 16, None, None)
    assert rc == pa.PA_ERR_INVALID
    assert np.prod([N, hq, S - 1, d + 1]) * 4 <= limit
