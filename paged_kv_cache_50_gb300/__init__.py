"""Python binding of libpa.so, the GB300 paged-attention library.

Argument marshalling only: each function checks that the torch tensors it is
given have the dtype, device and contiguity the C ABI (``include/pa.h``)
expects, passes their raw device pointers and the current CUDA stream, and
raises :class:`PaError` on a non-OK status.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback.  If ``libpa.so``
has not been built, every call raises.

Function names follow the C ABI: ``pa_reshape_and_cache``, ``pa_varlen_fwd``,
``pa_num_kv_splits``, ``pa_decode_workspace_bytes``, ``pa_decode_splitkv``,
``pa_lse_merge``, ``pa_mla_decode``, ``pa_get_device_error``.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA = 0, 1, 2, 3
PA_DEVERR_BLOCK_ID, PA_DEVERR_SLOT, PA_DEVERR_TIMEOUT, PA_DEVERR_LENGTH = 1, 2, 4, 8

_lock = threading.Lock()
_lib = None


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class PaShape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int), ("num_q_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_size", ctypes.c_int),
                ("block_size", ctypes.c_int), ("num_blocks", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int)]


def lib() -> ctypes.CDLL:
    """Loads libpa.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_50_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, f32, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int
        SP = ctypes.POINTER(PaShape)
        L.pa_reshape_and_cache.argtypes = [P, P, P, P, i32, SP, P]
        L.pa_varlen_fwd.argtypes = [P, P, P, P, P, i32, i32, SP, f32, i32, P, P, P]
        L.pa_num_kv_splits.argtypes = [i32, i32]
        L.pa_num_kv_splits.restype = i32
        L.pa_mla_num_kv_splits.argtypes = [i32, i32, i32, i32]
        L.pa_decode_num_kv_splits.argtypes = [i32, i32, i32, i32]
        L.pa_decode_num_kv_splits.restype = i32
        L.pa_mla_num_kv_splits.restype = i32
        L.pa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.pa_decode_workspace_bytes.restype = ctypes.c_size_t
        L.pa_decode_splitkv.argtypes = [P, P, P, P, SP, f32, i32, i32, P, P]
        L.pa_lse_merge.argtypes = [P, i32, i32, i32, i32, P, P, P]
        L.pa_varlen_fwd_window.argtypes = [P, P, P, P, P, i32, i32, SP, f32, i32, P, P, P]
        L.pa_cascade_fwd.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, SP, f32, i32,
                                     P, P, P, P]
        L.pa_cascade_prefix_splits.argtypes = [i32, i32, i32, i32, i32]
        L.pa_cascade_prefix_splits.restype = i32
        L.pa_reshape_and_cache_fp8.argtypes = [P, P, P, P, i32, SP, f32, f32, P]
        L.pa_mla_cache_write.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P]
        L.pa_mla_prefill_workspace_bytes.argtypes = [i32, i32, i32]
        L.pa_mla_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.pa_mla_expand_kv.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]
        L.pa_mla_prefill.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                     f32, i32, P, P, P, P]
        L.pa_decode_splitkv_fp8.argtypes = [P, P, P, P, SP, f32, f32, f32, i32, i32, P, P]
        L.pa_mla_decode.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                    i32, P, P, P, P]
        L.pa_decode_noalloc.argtypes = [P, P, P, P, SP, f32, i32, i32, P, P, P]
        L.pa_status_string.argtypes = [st]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), P]
        L.pa_device_sm_count.argtypes = []
        L.pa_device_sm_count.restype = i32
        for name in ("pa_reshape_and_cache", "pa_varlen_fwd", "pa_decode_splitkv",
                     "pa_lse_merge", "pa_mla_decode", "pa_get_device_error", "pa_decode_noalloc",
                     "pa_reshape_and_cache_fp8", "pa_decode_splitkv_fp8", "pa_varlen_fwd_window",
                     "pa_cascade_fwd", "pa_mla_cache_write", "pa_mla_expand_kv",
                     "pa_mla_prefill"):
            getattr(L, name).restype = st
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PaError(status, what)


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t, name, dtype):
    return None if t is None else _dev(t, name, dtype)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _pool_shape(kv_cache: torch.Tensor, num_seqs: int, num_q_heads: int,
                max_blocks: int) -> PaShape:
    if kv_cache.dim() != 5 or kv_cache.shape[1] != 2:
        raise ValueError("kv_cache must be [num_blocks, 2, block_size, num_kv_heads, head_size]")
    nb, _, bs, hkv, d = kv_cache.shape
    return PaShape(num_seqs, num_q_heads, hkv, d, bs, nb, max_blocks)


def pa_reshape_and_cache(key, value, kv_cache, slot_mapping, stream=None) -> None:
    """Writes key/value [T, Hkv, d] bf16 into kv_cache at slot_mapping [T] int64."""
    shape = _pool_shape(kv_cache, 0, kv_cache.shape[3], 1)
    T = key.shape[0]
    if tuple(key.shape) != (T, shape.num_kv_heads, shape.head_size) or value.shape != key.shape:
        raise ValueError("key/value must be [num_tokens, num_kv_heads, head_size]")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    _check(lib().pa_reshape_and_cache(
        _dev(key, "key", torch.bfloat16), _dev(value, "value", torch.bfloat16),
        _dev(kv_cache, "kv_cache", torch.bfloat16), _dev(slot_mapping, "slot_mapping", torch.int64),
        T, ctypes.byref(shape), _stream(stream)), "pa_reshape_and_cache")


def pa_mla_cache_write(kv_c, k_pe, kv_cache, slot_mapping, stream=None) -> None:
    """Writes [kv_c | k_pe] ([T, R], [T, P] bf16) into the MLA pool
    [nb, bs, R + P] at slot_mapping [T] int64."""
    if kv_cache.dim() != 3:
        raise ValueError("kv_cache must be [num_blocks, block_size, kv_lora_rank + rope_dim]")
    nb, bs, w = kv_cache.shape
    T, R = kv_c.shape
    if k_pe.dim() != 2 or k_pe.shape[0] != T or R + k_pe.shape[1] != w:
        raise ValueError("kv_c [T, R] and k_pe [T, P] must fill a cache row of R + P")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    _check(lib().pa_mla_cache_write(
        _dev(kv_c, "kv_c", torch.bfloat16), _dev(k_pe, "k_pe", torch.bfloat16),
        _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(slot_mapping, "slot_mapping", torch.int64), T, R, int(k_pe.shape[1]), bs, nb,
        _stream(stream)), "pa_mla_cache_write")


def mla_prefill_workspace(num_seqs, max_seq_len, num_heads, device="cuda"):
    """(k_ws [N, S, H, 192], v_ws [N, S, H, 128]) bf16 for the MLA prefill."""
    k = torch.empty((num_seqs, max_seq_len, num_heads, 192), dtype=torch.bfloat16, device=device)
    v = torch.empty((num_seqs, max_seq_len, num_heads, 128), dtype=torch.bfloat16, device=device)
    return k, v


def pa_mla_expand_kv(kv_cache, w_kv_b, block_table, seq_lens, k_ws, v_ws, stream=None) -> None:
    """MLA prefill step 1: per head [W_UK c | k_pe] and W_UV c of every context
    token into k_ws [N, S, H, 192] / v_ws [N, S, H, 128] (S = max_seq_len)."""
    nb, bs, w = kv_cache.shape
    H = w_kv_b.shape[0]
    N, S = k_ws.shape[0], k_ws.shape[1]
    if tuple(w_kv_b.shape) != (H, 256, 512) or w != 576:
        raise ValueError("w_kv_b must be [H, 256, 512] and kv_cache [nb, bs, 576]")
    if tuple(k_ws.shape) != (N, S, H, 192) or tuple(v_ws.shape) != (N, S, H, 128):
        raise ValueError("k_ws must be [N, S, H, 192] and v_ws [N, S, H, 128]")
    _check(lib().pa_mla_expand_kv(
        _dev(kv_cache, "kv_cache", torch.bfloat16), _dev(w_kv_b, "w_kv_b", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        N, H, bs, nb, int(block_table.shape[1]), S, _dev(k_ws, "k_ws", torch.bfloat16),
        _dev(v_ws, "v_ws", torch.bfloat16), _stream(stream)), "pa_mla_expand_kv")


def pa_mla_prefill_workspace_bytes(num_seqs, max_seq_len, num_heads) -> int:
    return int(lib().pa_mla_prefill_workspace_bytes(int(num_seqs), int(max_seq_len),
                                                    int(num_heads)))


def pa_mla_prefill(q, kv_cache, w_kv_b, block_table, query_start_loc, seq_lens, max_query_len,
                   scale, workspace, max_seq_len=None, causal=True, out=None, lse=None,
                   return_lse=True, stream=None):
    """MLA prefill (forward_mha): q [T, H, 192] against each request's latent
    context expanded through w_kv_b [H, 256, 512] -> (out [T, H, 128] bf16,
    lse [T, H] fp32).  ``workspace``: a uint8 tensor of at least
    pa_mla_prefill_workspace_bytes(N, max_seq_len, H) bytes."""
    T, H, dk = q.shape
    N = seq_lens.shape[0]
    nb, bs, w = kv_cache.shape
    if dk != 192 or w != 576 or tuple(w_kv_b.shape) != (H, 256, 512):
        raise ValueError("q [T, H, 192], kv_cache [nb, bs, 576], w_kv_b [H, 256, 512] expected")
    if query_start_loc.shape != (N + 1,) or block_table.dim() != 2 or block_table.shape[0] != N:
        raise ValueError("query_start_loc [N + 1] and block_table [N, max_blocks] expected")
    S = _max_seq(seq_lens, max_seq_len)
    need = pa_mla_prefill_workspace_bytes(N, S, H)
    if workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of at least {need} bytes")
    if out is None:
        out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    _check(lib().pa_mla_prefill(
        _dev(q, "q", torch.bfloat16), _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(w_kv_b, "w_kv_b", torch.bfloat16), _dev(block_table, "block_table", torch.int32),
        _dev(query_start_loc, "query_start_loc", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), T, int(max_query_len), N, H, bs, nb,
        int(block_table.shape[1]), S, float(scale), int(bool(causal)),
        _dev(workspace, "workspace", torch.uint8), _dev(out, "out", torch.bfloat16),
        _opt(lse, "lse", torch.float32), _stream(stream)), "pa_mla_prefill")
    return out, lse


def pa_varlen_fwd(q, kv_cache, block_table, query_start_loc, seq_lens, max_query_len, scale,
                  causal=True, out=None, lse=None, return_lse=True, stream=None):
    """Varlen paged attention.  q [T, Hq, d] bf16 -> (out [T, Hq, d] bf16,
    lse [T, Hq] fp32 or None)."""
    T, hq, d = q.shape
    N = seq_lens.shape[0]
    if query_start_loc.shape != (N + 1,):
        raise ValueError("query_start_loc must be [num_seqs + 1]")
    if block_table.dim() != 2 or block_table.shape[0] != N:
        raise ValueError("block_table must be [num_seqs, max_blocks]")
    shape = _pool_shape(kv_cache, N, hq, block_table.shape[1])
    if d != shape.head_size:
        raise ValueError("q head_size does not match kv_cache")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    _check(lib().pa_varlen_fwd(
        _dev(q, "q", torch.bfloat16), _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32),
        _dev(query_start_loc, "query_start_loc", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), T, int(max_query_len), ctypes.byref(shape),
        float(scale), int(bool(causal)), _dev(out, "out", torch.bfloat16),
        _opt(lse, "lse", torch.float32), _stream(stream)), "pa_varlen_fwd")
    return out, lse


def pa_varlen_fwd_window(q, kv_cache, block_table, query_start_loc, seq_lens, max_query_len,
                         scale, sliding_window, out=None, lse=None, return_lse=True, stream=None):
    """Causal varlen paged attention in which a row at position p sees only
    p - sliding_window < p' <= p.  Returns (out, lse) like pa_varlen_fwd."""
    T, hq, d = q.shape
    N = seq_lens.shape[0]
    if query_start_loc.shape != (N + 1,):
        raise ValueError("query_start_loc must be [num_seqs + 1]")
    if block_table.dim() != 2 or block_table.shape[0] != N:
        raise ValueError("block_table must be [num_seqs, max_blocks]")
    shape = _pool_shape(kv_cache, N, hq, block_table.shape[1])
    if d != shape.head_size:
        raise ValueError("q head_size does not match kv_cache")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    _check(lib().pa_varlen_fwd_window(
        _dev(q, "q", torch.bfloat16), _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32),
        _dev(query_start_loc, "query_start_loc", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), T, int(max_query_len), ctypes.byref(shape),
        float(scale), int(sliding_window), _dev(out, "out", torch.bfloat16),
        _opt(lse, "lse", torch.float32), _stream(stream)), "pa_varlen_fwd_window")
    return out, lse


def pa_cascade_prefix_splits(total_q, num_q_heads, num_kv_heads, prefix_tokens, sm_count=0):
    return int(lib().pa_cascade_prefix_splits(int(total_q), int(num_q_heads), int(num_kv_heads),
                                              int(prefix_tokens), int(sm_count)))


def cascade_workspace(total_q, num_q_heads, num_prefix_splits, num_suffix_splits, head_size,
                      device="cuda"):
    """fp32 [total_q, Hq, S1 + S2, d + 1] workspace for pa_cascade_fwd."""
    return torch.empty((total_q, num_q_heads, num_prefix_splits + num_suffix_splits,
                        head_size + 1), dtype=torch.float32, device=device)


def pa_cascade_fwd(q, kv_cache, block_table, query_start_loc, seq_lens, max_query_len,
                   num_common_prefix_blocks, scale, workspace, num_prefix_splits,
                   max_seq_len=None, causal=True, out=None, lse=None, return_lse=True,
                   stream=None):
    """Cascade attention: the shared first ``num_common_prefix_blocks`` blocks
    once for all rows (``num_prefix_splits`` pieces), each request's own
    blocks separately (the workspace's remaining slots), merged by LSE.
    ``workspace`` is [T, Hq, S1 + S2, d + 1] fp32 (see cascade_workspace)."""
    T, hq, d = q.shape
    N = seq_lens.shape[0]
    if query_start_loc.shape != (N + 1,):
        raise ValueError("query_start_loc must be [num_seqs + 1]")
    if block_table.dim() != 2 or block_table.shape[0] != N:
        raise ValueError("block_table must be [num_seqs, max_blocks]")
    shape = _pool_shape(kv_cache, N, hq, block_table.shape[1])
    if workspace.dim() != 4 or tuple(workspace.shape[:2]) != (T, hq) or \
            workspace.shape[3] != d + 1 or workspace.shape[2] <= int(num_prefix_splits):
        raise ValueError("workspace must be [total_q, num_q_heads, S1 + S2, d + 1] with S2 >= 1")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    s1 = int(num_prefix_splits)
    _check(lib().pa_cascade_fwd(
        _dev(q, "q", torch.bfloat16), _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32),
        _dev(query_start_loc, "query_start_loc", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32), T, int(max_query_len),
        _max_seq(seq_lens, max_seq_len), int(num_common_prefix_blocks), s1,
        int(workspace.shape[2]) - s1, ctypes.byref(shape), float(scale), int(bool(causal)),
        _dev(workspace, "workspace", torch.float32), _dev(out, "out", torch.bfloat16),
        _opt(lse, "lse", torch.float32), _stream(stream)), "pa_cascade_fwd")
    return out, lse


def pa_num_kv_splits(max_seq_len: int, sm_count: int = 0) -> int:
    return int(lib().pa_num_kv_splits(int(max_seq_len), int(sm_count)))


def pa_decode_num_kv_splits(num_seqs: int, num_kv_heads: int, max_seq_len: int,
                            sm_count: int = 0) -> int:
    return int(lib().pa_decode_num_kv_splits(int(num_seqs), int(num_kv_heads), int(max_seq_len),
                                             int(sm_count)))


def pa_mla_num_kv_splits(batch: int, num_heads: int, max_seq_len: int,
                         sm_count: int = 0) -> int:
    return int(lib().pa_mla_num_kv_splits(int(batch), int(num_heads), int(max_seq_len),
                                          int(sm_count)))


def pa_decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_splits: int, dv: int) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_splits, dv))


def pa_device_sm_count() -> int:
    return int(lib().pa_device_sm_count())


def decode_workspace(num_seqs, num_q_heads, num_splits, dv, device="cuda"):
    """Allocates a [N, Hq, S, dv + 1] fp32 split-KV workspace (torch owns it)."""
    return torch.empty((num_seqs, num_q_heads, num_splits, dv + 1), dtype=torch.float32,
                       device=device)


def _max_seq(seq_lens, max_seq_len):
    """The batch's longest seq_len; read from the device (a sync) only if the
    caller does not pass it."""
    if max_seq_len is not None:
        return int(max_seq_len)
    return int(seq_lens.max().item()) if seq_lens.numel() else 0


def pa_decode_splitkv(q, kv_cache, block_table, seq_lens, scale, workspace, max_seq_len=None,
                      stream=None) -> None:
    """Split-KV stage 1: q [N, Hq, d] -> workspace [N, Hq, S, d + 1] fp32.
    ``max_seq_len`` sizes the split chunk (default: read from ``seq_lens``)."""
    N, hq, d = q.shape
    if workspace.dim() != 4 or tuple(workspace.shape[:2]) != (N, hq) or workspace.shape[3] != d + 1:
        raise ValueError("workspace must be [num_seqs, num_q_heads, num_splits, head_size + 1]")
    shape = _pool_shape(kv_cache, N, hq, block_table.shape[1])
    _check(lib().pa_decode_splitkv(
        _dev(q, "q", torch.bfloat16), _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        ctypes.byref(shape), float(scale), int(workspace.shape[2]),
        _max_seq(seq_lens, max_seq_len), _dev(workspace, "workspace", torch.float32),
        _stream(stream)), "pa_decode_splitkv")


def _codes(kv_cache: torch.Tensor) -> torch.Tensor:
    """An fp8 pool as its bytes: uint8 codes, or float8_e4m3fn viewed as uint8."""
    if isinstance(kv_cache, torch.Tensor) and kv_cache.dtype == torch.float8_e4m3fn:
        return kv_cache.view(torch.uint8)
    return kv_cache


def pa_reshape_and_cache_fp8(key, value, kv_cache, slot_mapping, k_scale, v_scale,
                             stream=None) -> None:
    """Quantising cache write: key/value [T, Hkv, d] bf16 -> e4m3 codes of
    key / k_scale and value / v_scale in the fp8 pool kv_cache
    [nb, 2, bs, Hkv, d] (uint8 or float8_e4m3fn)."""
    codes = _codes(kv_cache)
    shape = _pool_shape(codes, 0, codes.shape[3], 1)
    T = key.shape[0]
    if tuple(key.shape) != (T, shape.num_kv_heads, shape.head_size) or value.shape != key.shape:
        raise ValueError("key/value must be [num_tokens, num_kv_heads, head_size]")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    _check(lib().pa_reshape_and_cache_fp8(
        _dev(key, "key", torch.bfloat16), _dev(value, "value", torch.bfloat16),
        _dev(codes, "kv_cache", torch.uint8), _dev(slot_mapping, "slot_mapping", torch.int64),
        T, ctypes.byref(shape), float(k_scale), float(v_scale), _stream(stream)),
        "pa_reshape_and_cache_fp8")


def pa_decode_splitkv_fp8(q, kv_cache, block_table, seq_lens, scale, k_scale, v_scale,
                          workspace, max_seq_len=None, stream=None) -> None:
    """Split-KV stage 1 over an fp8 pool (entries = e4m3 value x k_scale or
    v_scale): q [N, Hq, d] bf16 -> workspace [N, Hq, S, d + 1] fp32."""
    codes = _codes(kv_cache)
    N, hq, d = q.shape
    if workspace.dim() != 4 or tuple(workspace.shape[:2]) != (N, hq) or workspace.shape[3] != d + 1:
        raise ValueError("workspace must be [num_seqs, num_q_heads, num_splits, head_size + 1]")
    shape = _pool_shape(codes, N, hq, block_table.shape[1])
    _check(lib().pa_decode_splitkv_fp8(
        _dev(q, "q", torch.bfloat16), _dev(codes, "kv_cache", torch.uint8),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        ctypes.byref(shape), float(scale), float(k_scale), float(v_scale),
        int(workspace.shape[2]), _max_seq(seq_lens, max_seq_len),
        _dev(workspace, "workspace", torch.float32), _stream(stream)), "pa_decode_splitkv_fp8")


def pa_decode_fp8(q, kv_cache, block_table, seq_lens, scale, k_scale, v_scale, workspace,
                  out=None, lse=None, max_seq_len=None, stream=None):
    """Both split-KV stages over an fp8 pool."""
    pa_decode_splitkv_fp8(q, kv_cache, block_table, seq_lens, scale, k_scale, v_scale,
                          workspace, max_seq_len, stream)
    return pa_lse_merge(workspace, out, lse, stream=stream)


def pa_lse_merge(workspace, out=None, lse=None, return_lse=True, stream=None):
    """Split-KV stage 2: workspace [N, H, S, dv + 1] -> (out [N, H, dv] bf16, lse [N, H])."""
    N, H, S, dv1 = workspace.shape
    if out is None:
        out = torch.empty((N, H, dv1 - 1), dtype=torch.bfloat16, device=workspace.device)
    if lse is None and return_lse:
        lse = torch.empty((N, H), dtype=torch.float32, device=workspace.device)
    _check(lib().pa_lse_merge(
        _dev(workspace, "workspace", torch.float32), N, H, S, dv1 - 1,
        _dev(out, "out", torch.bfloat16), _opt(lse, "lse", torch.float32), _stream(stream)),
        "pa_lse_merge")
    return out, lse


def pa_decode(q, kv_cache, block_table, seq_lens, scale, workspace, out=None, lse=None,
              max_seq_len=None, stream=None):
    """Both split-KV stages: stage 1 into ``workspace``, then the LSE merge."""
    pa_decode_splitkv(q, kv_cache, block_table, seq_lens, scale, workspace, max_seq_len, stream)
    return pa_lse_merge(workspace, out, lse, stream=stream)


def pa_mla_decode(q, kv_cache, block_table, seq_lens, scale, workspace, out=None, lse=None,
                  kv_lora_rank=512, rope_dim=64, max_seq_len=None, stream=None):
    """MLA latent decode.  q [B, H, 576], kv_cache [nb, bs, 576] ->
    (out [B, H, 512] bf16, lse [B, H] fp32)."""
    B, H, dk = q.shape
    if kv_cache.dim() != 3 or kv_cache.shape[2] != dk or dk != kv_lora_rank + rope_dim:
        raise ValueError("kv_cache must be [num_blocks, block_size, kv_lora_rank + rope_dim]")
    if workspace.dim() != 4 or tuple(workspace.shape[:2]) != (B, H) or \
            workspace.shape[3] != kv_lora_rank + 1:
        raise ValueError("workspace must be [batch, num_heads, num_splits, kv_lora_rank + 1]")
    nb, bs, _ = kv_cache.shape
    if out is None:
        out = torch.empty((B, H, kv_lora_rank), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _check(lib().pa_mla_decode(
        _dev(q, "q", torch.bfloat16), _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        B, H, kv_lora_rank, rope_dim, bs, nb, block_table.shape[1],
        _max_seq(seq_lens, max_seq_len), float(scale), int(workspace.shape[2]),
        _dev(workspace, "workspace", torch.float32), _dev(out, "out", torch.bfloat16),
        _opt(lse, "lse", torch.float32), _stream(stream)), "pa_mla_decode")
    return out, lse


PA_NOALLOC_WORKSPACE_BYTES = 16 * 1024 * 1024


def pa_decode_noalloc(q, kv_cache, block_table, seq_lens, scale, num_splits, out=None,
                      lse=None, max_seq_len=None, stream=None):
    """Split-KV decode with the partials in the library's fixed device array
    (no workspace argument, nothing allocated by the library).  For callers
    that cannot allocate device memory; calls that overlap on the GPU race
    on the shared array.  ``out``/``lse`` are allocated here only if not
    given."""
    N, hq, d = q.shape
    shape = _pool_shape(kv_cache, N, hq, block_table.shape[1])
    if out is None:
        out = torch.empty((N, hq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((N, hq), dtype=torch.float32, device=q.device)
    _check(lib().pa_decode_noalloc(
        _dev(q, "q", torch.bfloat16), _dev(kv_cache, "kv_cache", torch.bfloat16),
        _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        ctypes.byref(shape), float(scale), int(num_splits), _max_seq(seq_lens, max_seq_len),
        _dev(out, "out", torch.bfloat16), _opt(lse, "lse", torch.float32), _stream(stream)),
        "pa_decode_noalloc")
    return out, lse


def pa_get_device_error(stream=None) -> int:
    """Synchronises the stream, returns and clears the PA_DEVERR_* bits."""
    code = ctypes.c_int(0)
    _check(lib().pa_get_device_error(ctypes.byref(code), _stream(stream)), "pa_get_device_error")
    return code.value
