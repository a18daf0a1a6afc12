"""Paged-attention oracle -- TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU implementation of the paged-attention hot path
(``pa_oracle.cpp``), loaded with ctypes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package.  It shares no code with ``paged_kv_cache_50_gb300`` and never
imports it; inputs come from the seeded generators in ``workloads``.

Every function takes numpy arrays (bf16 data as ``uint16`` bit patterns, or
``float64``) and returns fp64 results.  See ``pa_oracle.cpp`` for the
page-by-page citations and the readings taken where the pages are silent.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.cpp`` into ``_build/liboracle.so`` with g++."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, i64, i32, i32, i32, i64]
    lib.oracle_reshape_and_cache.restype = i32
    lib.oracle_mla_cache_write.argtypes = [P, P, P, P, i64, i32, i32, i32, i64]
    lib.oracle_mla_prefill.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                       i32, i64, f64, i32, i32, P, P, P, P, i32]
    lib.oracle_mla_prefill.restype = i32
    lib.oracle_round_bf16.argtypes = [P, P, i64]
    lib.oracle_round_bf16.restype = None
    lib.oracle_mla_cache_write.restype = i32
    for name in ("oracle_paged_attention_bf16", "oracle_paged_attention_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, i32, i64, f64,
                       i32, i32, P, P, P, i32]
        fn.restype = i32
    for name in ("oracle_split_partials_bf16", "oracle_split_partials_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f64,
                       i32, i64, P, i32]
        fn.restype = i32
    lib.oracle_lse_merge.argtypes = [P, i32, i32, i32, i32, P, P]
    lib.oracle_lse_merge.restype = None
    for name in ("oracle_mla_decode_bf16", "oracle_mla_decode_f64"):
        fn = getattr(lib, name)
        fn.argtypes = [P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f64,
                       P, P, P, i32]
        fn.restype = i32
    lib.oracle_bf16_to_f64.argtypes = [P, P, i64]
    lib.oracle_bf16_to_f64.restype = None
    lib.oracle_e4m3_decode.argtypes = [P, P, i64]
    lib.oracle_e4m3_decode.restype = None
    lib.oracle_e4m3_encode_f32.argtypes = [P, P, i64]
    lib.oracle_e4m3_encode_f32.restype = None
    lib.oracle_reshape_and_cache_fp8.argtypes = [P, P, P, P, i64, i32, i32, i32, i64,
                                                 ctypes.c_float, ctypes.c_float]
    lib.oracle_reshape_and_cache_fp8.restype = i32
    lib.oracle_dequant_pool_fp8.argtypes = [P, i64, i32, i32, i32, ctypes.c_float,
                                            ctypes.c_float, P]
    lib.oracle_dequant_pool_fp8.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def build_variant(source_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (the mutation tests plant
    deliberate slips this way to show that the pins catch them)."""
    src = out_path + ".cpp"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["g++", "-std=c++17", "-O1", "-fPIC", "-shared", "-pthread",
                    "-fno-fast-math", "-ffp-contract=off", src, "-o", out_path], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


@contextlib.contextmanager
def using_library(path: str):
    """Route every oracle call to another build of the source for a while."""
    global _lib
    old = _load()
    with _lock:
        _lib = _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = old


def default_threads() -> int:
    return os.cpu_count() or 1


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _kind(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return "bf16", a
    return "f64", np.ascontiguousarray(a, dtype=np.float64)


def reshape_and_cache(key, value, pool, slot_mapping, block_size):
    """Returns a copy of ``pool`` ([nb, 2, bs, Hkv, d] uint16) with the new
    key/value rows ([T, Hkv, d] uint16) written at ``slot_mapping`` [T]."""
    lib = _load()
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    out = np.array(pool, dtype=np.uint16, copy=True, order="C")
    slots = _c(slot_mapping, np.int64)
    T, Hkv, d = key.shape
    nb = out.shape[0]
    rc = lib.oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(out), _ptr(slots),
                                      T, Hkv, d, block_size, nb)
    if rc != 0:
        raise ValueError("slot outside the pool")
    return out


def mla_cache_write(kv_c, k_pe, pool, slot_mapping, block_size):
    """Returns a copy of the MLA pool ([nb, bs, R + P] uint16) with each new
    token's kv_c ([T, R]) and k_pe ([T, P]) written at ``slot_mapping`` [T]."""
    lib = _load()
    kv_c = _c(kv_c, np.uint16)
    k_pe = _c(k_pe, np.uint16)
    out = np.array(pool, dtype=np.uint16, copy=True, order="C")
    slots = _c(slot_mapping, np.int64)
    T, R = kv_c.shape
    P = k_pe.shape[1]
    assert out.shape[2] == R + P and k_pe.shape[0] == T
    rc = lib.oracle_mla_cache_write(_ptr(kv_c), _ptr(k_pe), _ptr(out), _ptr(slots), T, R, P,
                                    int(block_size), out.shape[0])
    if rc != 0:
        raise ValueError("slot outside the pool")
    return out


def mla_prefill(q, pool, w_kv_b, block_table, query_start_loc, seq_lens, scale, causal=True,
                round_kv=True, head_mask=None, row_mask=None, threads=None):
    """MLA prefill, multi-head formulation.  q [T, H, dn + dr], pool
    [nb, bs, R + dr], w_kv_b [H, dn + dv, R] (bf16 bits).  Each head's key is
    [w_kv_b[h, :dn] c | k_pe], its value w_kv_b[h, dn:] c (rounded to bf16
    with ``round_kv``).  Returns (out [T, H, dv], lse [T, H]) in fp64; rows or
    heads not selected by the masks are left at zero."""
    lib = _load()
    q = _c(q, np.uint16)
    pool = _c(pool, np.uint16)
    w = _c(w_kv_b, np.uint16)
    bt = _c(block_table, np.int32)
    qsl = _c(query_start_loc, np.int32)
    sl = _c(seq_lens, np.int32)
    T, H, dk = q.shape
    nb, bs, width = pool.shape
    Hw, wrow, R = w.shape
    assert Hw == H
    dr = width - R
    dn = dk - dr
    dv = wrow - dn
    out = np.zeros((T, H, dv), np.float64)
    lse = np.full((T, H), -np.inf, np.float64)
    hm = None if head_mask is None else _c(head_mask, np.uint8)
    rm = None if row_mask is None else _c(row_mask, np.uint8)
    rc = lib.oracle_mla_prefill(_ptr(q), _ptr(pool), _ptr(w), _ptr(bt), bt.shape[1], _ptr(qsl),
                                _ptr(sl), sl.shape[0], H, R, dr, dn, dv, bs, nb, float(scale),
                                int(bool(causal)), int(bool(round_kv)), _ptr(hm), _ptr(rm),
                                _ptr(out), _ptr(lse), threads or default_threads())
    if rc != 0:
        raise ValueError("invalid MLA prefill input")
    return out, lse


def round_bf16(x):
    """Nearest bf16 values (ties to even) of float64 values, as float64."""
    lib = _load()
    xs = _c(x, np.float64)
    out = np.empty(xs.shape, np.float64)
    lib.oracle_round_bf16(_ptr(xs), _ptr(out), xs.size)
    return out


def paged_attention(q, pool, block_table, query_start_loc, seq_lens, scale,
                    causal=True, row_mask=None, threads=None, window=0):
    """Varlen paged attention.  q [T, Hq, d]; pool [nb, 2, bs, Hkv, d]
    (uint16 bf16 bits, or float64).  Returns (out [T, Hq, d], lse [T, Hq])
    in fp64; rows not selected by ``row_mask`` are left at zero.
    ``window`` > 0 (causal only): a row at position p sees p - window < p' <= p."""
    lib = _load()
    kq, q = _kind(q)
    kp, pool = _kind(pool)
    if kq != kp:
        raise TypeError("q and pool must both be bf16 bits or both float64")
    q = np.ascontiguousarray(q)
    pool = np.ascontiguousarray(pool)
    bt = _c(block_table, np.int32)
    qsl = _c(query_start_loc, np.int32)
    sl = _c(seq_lens, np.int32)
    T, Hq, d = q.shape
    nb, two, bs, Hkv, d2 = pool.shape
    assert two == 2 and d2 == d
    N = sl.shape[0]
    out = np.zeros((T, Hq, d), np.float64)
    lse = np.full((T, Hq), -np.inf, np.float64)
    mask = None if row_mask is None else _c(row_mask, np.uint8)
    fn = lib.oracle_paged_attention_bf16 if kq == "bf16" else lib.oracle_paged_attention_f64
    rc = fn(_ptr(q), _ptr(pool), _ptr(bt), bt.shape[1], _ptr(qsl), _ptr(sl), N, Hq,
            Hkv, d, bs, nb, float(scale), int(bool(causal)), int(window), _ptr(mask),
            _ptr(out), _ptr(lse), threads or default_threads())
    if rc != 0:
        raise ValueError("invalid paged-attention input (block id, lengths or window)")
    return out, lse


def split_partials(q, pool, block_table, seq_lens, scale, num_splits, max_seq_len=None,
                   threads=None):
    """Split-KV stage 1 for one query per request.  q [N, Hq, d].
    Returns partials [N, Hq, S, d + 1] fp64 (normalised o, then lse).
    ``max_seq_len`` (default: the batch maximum) sizes the split chunk."""
    lib = _load()
    kq, q = _kind(q)
    kp, pool = _kind(pool)
    if kq != kp:
        raise TypeError("q and pool must both be bf16 bits or both float64")
    q = np.ascontiguousarray(q)
    pool = np.ascontiguousarray(pool)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    N, Hq, d = q.shape
    nb, _, bs, Hkv, _ = pool.shape
    out = np.zeros((N, Hq, num_splits, d + 1), np.float64)
    if max_seq_len is None:
        max_seq_len = int(sl.max()) if sl.size else 0
    fn = lib.oracle_split_partials_bf16 if kq == "bf16" else lib.oracle_split_partials_f64
    rc = fn(_ptr(q), _ptr(pool), _ptr(bt), bt.shape[1], _ptr(sl), N, Hq, Hkv, d, bs,
            nb, float(scale), int(num_splits), int(max_seq_len), _ptr(out),
            threads or default_threads())
    if rc != 0:
        raise ValueError("invalid split-KV input")
    return out


def lse_merge(partials):
    """Split-KV stage 2.  partials [N, H, S, dv + 1] -> (out [N, H, dv], lse [N, H])."""
    lib = _load()
    p = _c(partials, np.float64)
    N, H, S, dv1 = p.shape
    out = np.zeros((N, H, dv1 - 1), np.float64)
    lse = np.zeros((N, H), np.float64)
    lib.oracle_lse_merge(_ptr(p), N, H, S, dv1 - 1, _ptr(out), _ptr(lse))
    return out, lse


def mla_decode(q, pool, block_table, seq_lens, scale, kv_lora_rank=512,
               rope_dim=64, req_mask=None, threads=None):
    """MLA latent decode.  q [B, H, kv_lora_rank + rope_dim];
    pool [nb, bs, kv_lora_rank + rope_dim].  Returns (out [B, H, kv_lora_rank],
    lse [B, H]) fp64; requests not in ``req_mask`` are left at zero."""
    lib = _load()
    kq, q = _kind(q)
    kp, pool = _kind(pool)
    if kq != kp:
        raise TypeError("q and pool must both be bf16 bits or both float64")
    q = np.ascontiguousarray(q)
    pool = np.ascontiguousarray(pool)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    B, H, dk = q.shape
    nb, bs, dk2 = pool.shape
    assert dk == dk2 == kv_lora_rank + rope_dim
    out = np.zeros((B, H, kv_lora_rank), np.float64)
    lse = np.full((B, H), -np.inf, np.float64)
    mask = None if req_mask is None else _c(req_mask, np.uint8)
    fn = lib.oracle_mla_decode_bf16 if kq == "bf16" else lib.oracle_mla_decode_f64
    rc = fn(_ptr(q), _ptr(pool), _ptr(bt), bt.shape[1], _ptr(sl), B, H, kv_lora_rank,
            rope_dim, bs, nb, float(scale), _ptr(mask), _ptr(out), _ptr(lse),
            threads or default_threads())
    if rc != 0:
        raise ValueError("invalid MLA input (block id)")
    return out, lse


def bf16_to_f64(bits):
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    lib = _load()
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    lib.oracle_bf16_to_f64(_ptr(b), _ptr(out), b.size)
    return out


# ---------------------------------------------------------------- fp8 cache

def e4m3_decode(codes):
    """Values of e4m3 codes (uint8 array) as float64 (NaN for the NaN codes)."""
    lib = _load()
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib.oracle_e4m3_decode(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(x):
    """Nearest e4m3 codes (ties to even, saturating at +-448) of float32 values."""
    lib = _load()
    xs = _c(x, np.float32)
    out = np.empty(xs.shape, np.uint8)
    lib.oracle_e4m3_encode_f32(_ptr(xs), _ptr(out), xs.size)
    return out


def reshape_and_cache_fp8(key, value, pool, slot_mapping, block_size, k_scale, v_scale):
    """Step 1 into an fp8 pool: key/value [T, Hkv, d] bf16 bits, pool
    [nb, 2, bs, Hkv, d] uint8 e4m3 codes.  Returns the updated pool (a copy)."""
    lib = _load()
    k = _c(key, np.uint16)
    v = _c(value, np.uint16)
    out = np.array(pool, dtype=np.uint8, copy=True, order="C")
    sm = _c(slot_mapping, np.int64)
    T, Hkv, d = k.shape
    nb = out.shape[0]
    rc = lib.oracle_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(out), _ptr(sm), T, Hkv, d,
                                          int(block_size), nb, float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError("slot outside the pool")
    return out


def dequant_pool_fp8(pool, k_scale, v_scale):
    """Values of an fp8 pool [nb, 2, bs, Hkv, d]: K codes times k_scale, V
    codes times v_scale, as float64."""
    lib = _load()
    p = _c(pool, np.uint8)
    nb, two, bs, Hkv, d = p.shape
    out = np.empty(p.shape, np.float64)
    lib.oracle_dequant_pool_fp8(_ptr(p), nb, bs, Hkv, d, float(k_scale), float(v_scale),
                                _ptr(out))
    return out


def split_partials_fp8(q, pool, block_table, seq_lens, scale, k_scale, v_scale, num_splits,
                       max_seq_len=None, threads=None):
    """split_partials over the values of an fp8 pool (q: bf16 bits)."""
    return split_partials(bf16_to_f64(q), dequant_pool_fp8(pool, k_scale, v_scale), block_table,
                          seq_lens, scale, num_splits, max_seq_len=max_seq_len, threads=threads)
