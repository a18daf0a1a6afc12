"""Host-side checks of the C-ABI boundary (no GPU needed): the library loads,
exports every entry point ``include/pa.h`` declares, plans splits by the
page's rule, and rejects bad arguments before any launch."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def pa():
    from paged_kv_cache_50_gb300 import build
    build.build()
    import paged_kv_cache_50_gb300 as pa
    pa.lib()
    return pa


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_contract():
    names = _declared()
    for n in ("pa_reshape_and_cache", "pa_varlen_fwd", "pa_decode_splitkv", "pa_lse_merge",
              "pa_mla_decode", "pa_num_kv_splits", "pa_decode_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(pa):
    L = pa.lib()
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing


def test_split_rule_of_the_page(pa):
    # min(ceil(max_seq / 512), 2 * SMs), at least 1 ("Triton and MLA", key files).
    assert pa.pa_num_kv_splits(131072, 152) == 256
    assert pa.pa_num_kv_splits(131072, 100) == 200
    assert pa.pa_num_kv_splits(4096, 152) == 8
    assert pa.pa_num_kv_splits(4097, 152) == 9
    assert pa.pa_num_kv_splits(1, 152) == 1
    assert pa.pa_num_kv_splits(0, 152) == 1


def test_decode_split_planner(pa):
    # S = min(max(1, ceil(12 * SMs / (N * Hkv))), page rule): ~12 CTAs per SM.
    assert pa.pa_decode_num_kv_splits(64, 8, 4096, 152) == 4       # the GQA decode batch
    assert pa.pa_decode_num_kv_splits(8, 8, 131072, 152) == 29     # long context (the page: 256)
    assert pa.pa_decode_num_kv_splits(64, 8, 1000, 152) == 2       # capped by ceil(1000 / 512)
    assert pa.pa_decode_num_kv_splits(4096, 8, 4096, 152) == 1
    assert pa.pa_decode_num_kv_splits(1, 1, 1 << 20, 152) == 304   # capped at 2 x SMs
    assert pa.pa_decode_num_kv_splits(0, 8, 4096, 152) == 1
    assert pa.pa_decode_num_kv_splits(64, 8, 0, 152) == 1


def test_mla_split_planner(pa):
    # S = min(ceil((SMs / 2) / (batch * ceil(H / 128))), ceil(max_seq / 512)), at least 1:
    # one (split, request, head group) unit per SM pair, never finer than 512 tokens.
    assert pa.pa_mla_num_kv_splits(128, 128, 8192, 152) == 1      # the DeepSeek-V3-shape batch
    assert pa.pa_mla_num_kv_splits(8, 128, 8192, 152) == 10       # ceil(76 / 8)
    assert pa.pa_mla_num_kv_splits(8, 256, 8192, 152) == 5        # two head groups per request
    assert pa.pa_mla_num_kv_splits(1, 128, 131072, 152) == 76     # one request: every pair
    assert pa.pa_mla_num_kv_splits(1, 128, 2048, 152) == 4        # capped at 512-token pieces
    assert pa.pa_mla_num_kv_splits(1, 64, 100, 152) == 1
    assert pa.pa_mla_num_kv_splits(76, 128, 8192, 152) == 1
    assert pa.pa_mla_num_kv_splits(75, 128, 8192, 152) == 2
    assert pa.pa_mla_num_kv_splits(4, 128, 0, 152) == 1
    assert pa.pa_mla_num_kv_splits(0, 128, 4096, 152) == 1
    assert pa.pa_mla_num_kv_splits(2, 128, 1 << 20, 1) == 1      # fewer than two SMs


def test_workspace_bytes(pa):
    assert pa.pa_decode_workspace_bytes(8, 64, 256, 128) == 8 * 64 * 256 * 129 * 4
    assert pa.pa_decode_workspace_bytes(128, 128, 4, 512) == 128 * 128 * 4 * 513 * 4
    assert pa.pa_decode_workspace_bytes(0, 1, 1, 1) == 0
    assert pa.pa_decode_workspace_bytes(1, 1, 0, 1) == 0


def _shape(pa, **kw):
    base = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_size=128, block_size=16,
                num_blocks=10, max_blocks_per_seq=4)
    base.update(kw)
    return pa.PaShape(**base)


NULL = None


@pytest.mark.parametrize("kw,expect", [
    (dict(block_size=8), 1),        # block_size must be a multiple of 16
    (dict(block_size=0), 1),
    (dict(num_q_heads=6, num_kv_heads=4), 1),   # Hq % Hkv
    (dict(num_blocks=0), 1),
    (dict(head_size=96), 2),        # not built
    (dict(head_size=256), 2),
])
def test_varlen_rejects_bad_shapes_before_launch(pa, kw, expect):
    s = _shape(pa, **kw)
    rc = pa.lib().pa_varlen_fwd(1, 1, 1, 1, 1, 4, 2, ctypes.byref(s), 0.1, 1, 1, NULL, NULL)
    assert rc == expect


def test_varlen_rejects_null_pointers(pa):
    s = _shape(pa)
    assert pa.lib().pa_varlen_fwd(NULL, 1, 1, 1, 1, 4, 2, ctypes.byref(s), 0.1, 1, 1,
                                  NULL, NULL) == pa.PA_ERR_INVALID
    assert pa.lib().pa_varlen_fwd(1, 1, 1, 1, 1, 4, 2, None, 0.1, 1, 1, NULL, NULL) == \
        pa.PA_ERR_INVALID


def test_empty_calls_are_noops(pa):
    s = _shape(pa)
    assert pa.lib().pa_varlen_fwd(NULL, NULL, NULL, NULL, NULL, 0, 0, ctypes.byref(s), 0.1, 1,
                                  NULL, NULL, NULL) == pa.PA_OK
    assert pa.lib().pa_reshape_and_cache(NULL, NULL, NULL, NULL, 0, ctypes.byref(s),
                                         NULL) == pa.PA_OK
    s0 = _shape(pa, num_seqs=0)
    assert pa.lib().pa_decode_splitkv(NULL, NULL, NULL, NULL, ctypes.byref(s0), 0.1, 4, 0, NULL,
                                      NULL) == pa.PA_OK


def test_decode_rejects(pa):
    L = pa.lib()
    s = _shape(pa)
    assert L.pa_decode_splitkv(1, 1, 1, 1, ctypes.byref(s), 0.1, 0, 64, 1, NULL) == pa.PA_ERR_INVALID
    assert L.pa_decode_splitkv(1, 1, 1, 1, ctypes.byref(s), 0.1, 20000, 64, 1, NULL) == \
        pa.PA_ERR_INVALID
    big_group = _shape(pa, num_q_heads=64, num_kv_heads=2)
    assert L.pa_decode_splitkv(1, 1, 1, 1, ctypes.byref(big_group), 0.1, 4, 64, 1, NULL) == \
        pa.PA_ERR_UNSUPPORTED
    assert L.pa_decode_splitkv(1, 1, 1, 1, ctypes.byref(s), 0.1, 4, 64, NULL, NULL) == \
        pa.PA_ERR_INVALID
    assert L.pa_lse_merge(1, 2, 8, 0, 128, 1, NULL, NULL) == pa.PA_ERR_INVALID
    assert L.pa_lse_merge(NULL, 2, 8, 4, 128, 1, NULL, NULL) == pa.PA_ERR_INVALID


def test_limits_are_rejected_one_past(pa):
    """One past each launch limit: 65536 requests, 16385 splits."""
    L = pa.lib()
    s = _shape(pa, num_seqs=65536)
    assert L.pa_decode_splitkv(16, 16, 16, 16, ctypes.byref(s), 0.1, 4, 64, 16, NULL) == \
        pa.PA_ERR_INVALID
    assert L.pa_varlen_fwd(16, 16, 16, 16, 16, 1, 1, ctypes.byref(s), 0.1, 1, 16, NULL, NULL) == \
        pa.PA_ERR_INVALID
    ok = _shape(pa)
    assert L.pa_decode_splitkv(16, 16, 16, 16, ctypes.byref(ok), 0.1, 16385, 64, 16, NULL) == \
        pa.PA_ERR_INVALID
    assert L.pa_lse_merge(16, 2, 8, 16385, 128, 16, NULL, NULL) == pa.PA_ERR_INVALID
    assert L.pa_mla_decode(16, 16, 16, 16, 65536, 128, 512, 64, 64, 10, 10, 64, 0.1, 1, 16, 16,
                           NULL, NULL) == pa.PA_ERR_INVALID


def test_cache_write_rejects(pa):
    L = pa.lib()
    assert L.pa_reshape_and_cache(1, 1, 1, 1, 4, ctypes.byref(_shape(pa, block_size=24)),
                                  NULL) == pa.PA_ERR_INVALID
    assert L.pa_reshape_and_cache(1, 1, 1, 1, 4, ctypes.byref(_shape(pa, head_size=12)),
                                  NULL) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_reshape_and_cache(1, NULL, 1, 1, 4, ctypes.byref(_shape(pa)),
                                  NULL) == pa.PA_ERR_INVALID


def test_mla_rejects(pa):
    L = pa.lib()
    args = dict(batch=2, num_heads=128, kv_lora_rank=512, rope_dim=64, block_size=64,
                num_blocks=8, max_blocks=4, scale=0.07, num_splits=2)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.pa_mla_decode(1, 1, 1, 1, a["batch"], a["num_heads"], a["kv_lora_rank"],
                               a["rope_dim"], a["block_size"], a["num_blocks"], a["max_blocks"], 256,
                               a["scale"], a["num_splits"], 1, 1, NULL, NULL)
    assert call(kv_lora_rank=448) == pa.PA_ERR_UNSUPPORTED   # head sizes other than 576
    assert call(rope_dim=32) == pa.PA_ERR_UNSUPPORTED
    assert call(num_heads=40) == pa.PA_ERR_UNSUPPORTED
    assert call(block_size=48) == pa.PA_ERR_UNSUPPORTED
    assert call(block_size=8) == pa.PA_ERR_INVALID
    assert call(num_splits=0) == pa.PA_ERR_INVALID
    assert call(batch=0) == pa.PA_OK


def test_status_strings(pa):
    for st in range(4):
        assert pa.status_string(st).startswith("PA_")


def test_python_binding_refuses_cpu_tensors(pa):
    import torch
    kv = torch.zeros(4, 2, 16, 2, 64, dtype=torch.bfloat16)
    key = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    slots = torch.zeros(3, dtype=torch.int64)
    with pytest.raises(ValueError):
        pa.pa_reshape_and_cache(key, key, kv, slots)


def test_misaligned_pointers_are_rejected(pa):
    L = pa.lib()
    s = _shape(pa)
    # kv_cache must be 16-byte aligned (16-byte vector loads of cache rows).
    assert L.pa_varlen_fwd(16, 8, 16, 16, 16, 4, 2, ctypes.byref(s), 0.1, 1, 16, NULL,
                           NULL) == pa.PA_ERR_INVALID
    assert L.pa_reshape_and_cache(16, 24, 16, 16, 4, ctypes.byref(s), NULL) == pa.PA_ERR_INVALID
    assert L.pa_mla_decode(8, 16, 16, 16, 2, 128, 512, 64, 64, 8, 4, 256, 0.1, 2, 16, 16, NULL,
                           NULL) == pa.PA_ERR_INVALID


def test_fp8_entry_points_reject_before_launch(pa):
    L = pa.lib()
    s = _shape(pa)
    inf = float("inf")
    for ks, vs in ((0.0, 1.0), (1.0, -2.0), (inf, 1.0), (1.0, float("nan"))):
        assert L.pa_reshape_and_cache_fp8(16, 16, 16, 16, 4, ctypes.byref(s), ks, vs,
                                          NULL) == pa.PA_ERR_INVALID
        assert L.pa_decode_splitkv_fp8(16, 16, 16, 16, ctypes.byref(s), 0.1, ks, vs, 4, 64, 16,
                                       NULL) == pa.PA_ERR_INVALID
    # Codes move in 16-byte vectors: head sizes that are not a multiple of 16.
    assert L.pa_reshape_and_cache_fp8(16, 16, 16, 16, 4, ctypes.byref(_shape(pa, head_size=24)),
                                      1.0, 1.0, NULL) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_decode_splitkv_fp8(16, 16, 16, 16, ctypes.byref(_shape(pa, head_size=96)), 0.1,
                                   1.0, 1.0, 4, 64, 16, NULL) == pa.PA_ERR_UNSUPPORTED
    big_group = _shape(pa, num_q_heads=64, num_kv_heads=2)
    assert L.pa_decode_splitkv_fp8(16, 16, 16, 16, ctypes.byref(big_group), 0.1, 1.0, 1.0, 4, 64,
                                   16, NULL) == pa.PA_ERR_UNSUPPORTED
    # Misaligned pool, null workspace, bad split counts.
    assert L.pa_reshape_and_cache_fp8(16, 16, 24, 16, 4, ctypes.byref(s), 1.0, 1.0,
                                      NULL) == pa.PA_ERR_INVALID
    assert L.pa_decode_splitkv_fp8(16, 24, 16, 16, ctypes.byref(s), 0.1, 1.0, 1.0, 4, 64, 16,
                                   NULL) == pa.PA_ERR_INVALID
    assert L.pa_decode_splitkv_fp8(16, 16, 16, 16, ctypes.byref(s), 0.1, 1.0, 1.0, 4, 64, NULL,
                                   NULL) == pa.PA_ERR_INVALID
    assert L.pa_decode_splitkv_fp8(16, 16, 16, 16, ctypes.byref(s), 0.1, 1.0, 1.0, 0, 64, 16,
                                   NULL) == pa.PA_ERR_INVALID
    # Empty calls launch nothing.
    assert L.pa_reshape_and_cache_fp8(NULL, NULL, NULL, NULL, 0, ctypes.byref(s), 1.0, 1.0,
                                      NULL) == pa.PA_OK
    assert L.pa_decode_splitkv_fp8(NULL, NULL, NULL, NULL, ctypes.byref(_shape(pa, num_seqs=0)),
                                   0.1, 1.0, 1.0, 4, 64, NULL, NULL) == pa.PA_OK


def test_mla_cache_write_rejects(pa):
    L = pa.lib()
    assert L.pa_mla_cache_write(16, 16, 16, 16, 4, 512, 64, 24, 8, NULL) == pa.PA_ERR_INVALID
    assert L.pa_mla_cache_write(16, 16, 16, 16, 4, 500, 64, 64, 8, NULL) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_mla_cache_write(16, 16, 24, 16, 4, 512, 64, 64, 8, NULL) == pa.PA_ERR_INVALID
    assert L.pa_mla_cache_write(NULL, 16, 16, 16, 4, 512, 64, 64, 8, NULL) == pa.PA_ERR_INVALID
    assert L.pa_mla_cache_write(NULL, NULL, NULL, NULL, 0, 512, 64, 64, 8, NULL) == pa.PA_OK


def test_mla_prefill_workspace_alignment(pa):
    # The expansion writes workspace rows with 32-byte stores: 16-byte
    # aligned workspaces are refused before anything is launched.
    L = pa.lib()
    assert L.pa_mla_expand_kv(16, 16, 16, 16, 2, 16, 64, 8, 4, 100, 48, 64, NULL) == \
        pa.PA_ERR_INVALID
    assert L.pa_mla_expand_kv(16, 16, 16, 16, 2, 16, 64, 8, 4, 100, 64, 80, NULL) == \
        pa.PA_ERR_INVALID
    assert L.pa_mla_prefill(16, 16, 16, 16, 16, 16, 8, 4, 2, 16, 64, 8, 4, 100, 0.1, 1, 48, 16,
                            NULL, NULL) == pa.PA_ERR_INVALID


def test_window_and_cascade_reject(pa):
    L = pa.lib()
    s = _shape(pa)
    assert L.pa_varlen_fwd_window(16, 16, 16, 16, 16, 4, 2, ctypes.byref(s), 0.1, 0, 16, NULL,
                                  NULL) == pa.PA_ERR_INVALID          # window < 1
    assert L.pa_varlen_fwd_window(16, 16, 16, 16, 16, 4, 2, ctypes.byref(_shape(pa, head_size=96)),
                                  0.1, 8, 16, NULL, NULL) == pa.PA_ERR_UNSUPPORTED
    args = [16, 16, 16, 16, 16, 4, 2, 64]
    # num_common_prefix_blocks past the table, zero splits, too many splits.
    assert L.pa_cascade_fwd(*args, 5, 1, 1, ctypes.byref(s), 0.1, 1, 16, 16, NULL,
                            NULL) == pa.PA_ERR_INVALID
    assert L.pa_cascade_fwd(*args, 2, 0, 1, ctypes.byref(s), 0.1, 1, 16, 16, NULL,
                            NULL) == pa.PA_ERR_INVALID
    assert L.pa_cascade_fwd(*args, 2, 1, 0, ctypes.byref(s), 0.1, 1, 16, 16, NULL,
                            NULL) == pa.PA_ERR_INVALID
    assert L.pa_cascade_fwd(*args, 2, 10000, 10000, ctypes.byref(s), 0.1, 1, 16, 16, NULL,
                            NULL) == pa.PA_ERR_INVALID
    assert L.pa_cascade_fwd(*args, 2, 1, 1, ctypes.byref(s), 0.1, 1, NULL, 16, NULL,
                            NULL) == pa.PA_ERR_INVALID          # no workspace
    assert pa.pa_cascade_prefix_splits(64, 32, 8, 4096, 152) == 19
    assert pa.pa_cascade_prefix_splits(64, 32, 8, 128, 152) == 1   # one tile of prefix
    assert pa.pa_cascade_prefix_splits(0, 32, 8, 4096, 152) == 1
