"""Seeded synthetic inputs for the paged-attention hot path.

This module only draws random inputs and lays them out; it holds none of the
attention arithmetic.  Both sides of every parity check -- the CUDA library
and the fp64 oracle -- consume the arrays it returns, and neither side
imports the other.

Recipe (the same for every workload):
  * numpy ``default_rng(seed)`` draws N(0, 1) float32 values, rounded to bf16
    (round to nearest even) and kept as uint16 bit patterns; arrays of more
    than 2^22 values are drawn in 2^22-value chunks, chunk k from the k-th
    child generator (``Generator.spawn``);
  * request lengths are integers drawn uniformly from inclusive ranges;
  * the pool holds exactly sum_i ceil(seq_i / bs) blocks (unless a size is
    given); a seeded permutation of the block ids is handed out to the
    requests in order, so each request's blocks are scattered through the pool;
  * the whole pool is first filled with N(0, 1) values, then the step's new
    K/V (the last ``query_len`` positions of each request) are drawn and the
    slot of each new token is slot = block_table[i][pos // bs] * bs + pos % bs
    ("Attention Backends", section "Code");
  * entries of ``block_table`` past a request's last block are -1, so a kernel
    that read them would be caught;
  * an fp8 pool (same shape, one byte per element) is filled with uniformly
    random finite e4m3 codes; its scales are the fixed FP8_K_SCALE and
    FP8_V_SCALE.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _chunked_fill(rng: np.random.Generator, n: int, chunk: int, fill) -> None:
    """Calls fill(gen, a, m) for the chunks [a, a + m) of n elements.  An
    array of one chunk is drawn from ``rng`` itself; a larger one takes one
    child generator of ``rng`` per chunk (``Generator.spawn``, in chunk
    order), so the values do not depend on how many threads draw them, and
    the chunks are drawn on all host cores (numpy releases the GIL while it
    fills a buffer)."""
    if n <= chunk:
        fill(rng, 0, n)
        return
    starts = list(range(0, n, chunk))
    kids = rng.spawn(len(starts))
    work = [(kids[k], a, min(n, a + chunk) - a) for k, a in enumerate(starts)]
    threads = max(1, min(len(work), os.cpu_count() or 1))
    if threads == 1:
        for w in work:
            fill(*w)
        return
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda w: fill(*w), work))


def randn_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 22) -> np.ndarray:
    """N(0, 1) values rounded to bf16 (nearest even), as uint16 bits.  Drawn
    in chunks of ``chunk`` values (see _chunked_fill), so multi-GB pools need
    no float32 copy of the whole array."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)

    def fill(gen, a, m):
        f = np.empty(m, np.float32)
        gen.standard_normal(m, dtype=np.float32, out=f)
        u = f.view(np.uint32)
        t = np.right_shift(u, 16)
        t &= 1
        t += 0x7FFF
        t += u
        t >>= 16
        out[a:a + m] = t

    _chunked_fill(rng, n, chunk, fill)
    return out.reshape(shape)


@dataclass
class PagedBatch:
    """One step of the standard-layout workload (pool [nb, 2, bs, Hkv, d])."""
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray          # int32 [N]
    query_lens: np.ndarray        # int32 [N]
    query_start_loc: np.ndarray   # int32 [N + 1]
    block_table: np.ndarray       # int32 [N, max_blocks], -1 past the end
    slot_mapping: np.ndarray      # int64 [T]
    q: np.ndarray                 # uint16 [T, Hq, d]
    key: np.ndarray               # uint16 [T, Hkv, d] (new tokens)
    value: np.ndarray             # uint16 [T, Hkv, d]
    pool: np.ndarray              # uint16 [nb, 2, bs, Hkv, d] BEFORE the write
    scale: float
    causal: bool = True
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def kv_bytes(self) -> int:
        """Bytes of K and V a decode pass must read (bf16)."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_size * 2 * 2

    def causal_flops(self) -> int:
        """4 * d * Hq * sum_i(qlen_i * ctx_i + qlen_i (qlen_i + 1) / 2)."""
        ql = self.query_lens.astype(np.int64)
        ctx = self.seq_lens.astype(np.int64) - ql
        pairs = int((ql * ctx + ql * (ql + 1) // 2).sum())
        return 4 * self.head_size * self.num_q_heads * pairs


def _assign_blocks(rng, seq_lens, block_size, num_blocks=None):
    need = [(int(s) + block_size - 1) // block_size for s in seq_lens]
    total = sum(need)
    nb = total if num_blocks is None else int(num_blocks)
    if nb < total:
        raise ValueError("pool too small")
    perm = rng.permutation(nb).astype(np.int32)
    max_blocks = max(1, max(need) if need else 1)
    table = np.full((len(seq_lens), max_blocks), -1, np.int32)
    k = 0
    for i, n in enumerate(need):
        table[i, :n] = perm[k:k + n]
        k += n
    return table, nb


def make_paged_batch(name, seed, seq_lens, query_lens, num_q_heads, num_kv_heads,
                     head_size, block_size, num_blocks=None, scale=None,
                     causal=True, with_pool=True) -> PagedBatch:
    """with_pool=False skips drawing the pool (``pool`` is None); the other
    arrays are drawn exactly as with the pool, from a separate stream."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    query_lens = np.asarray(query_lens, np.int32)
    assert np.all(query_lens <= seq_lens) and np.all(query_lens >= 0)
    N = seq_lens.shape[0]
    qsl = np.zeros(N + 1, np.int32)
    qsl[1:] = np.cumsum(query_lens)
    table, nb = _assign_blocks(rng, seq_lens, block_size, num_blocks)
    T = int(qsl[-1])
    slots = np.empty(T, np.int64)
    for i in range(N):
        ctx = int(seq_lens[i] - query_lens[i])
        for j in range(int(query_lens[i])):
            pos = ctx + j
            slots[qsl[i] + j] = int(table[i, pos // block_size]) * block_size + pos % block_size
    pool = randn_bf16(rng, (nb, 2, block_size, num_kv_heads, head_size)) if with_pool else None
    rng = np.random.default_rng([seed, 1])
    q = randn_bf16(rng, (T, num_q_heads, head_size))
    key = randn_bf16(rng, (T, num_kv_heads, head_size))
    value = randn_bf16(rng, (T, num_kv_heads, head_size))
    if scale is None:
        scale = 1.0 / math.sqrt(head_size)
    return PagedBatch(name, seed, num_q_heads, num_kv_heads, head_size, block_size, nb,
                      seq_lens, query_lens, qsl, table, slots, q, key, value, pool,
                      float(scale), causal)


@dataclass
class MLABatch:
    """One decode step of the MLA latent workload (pool [nb, bs, 576])."""
    name: str
    seed: int
    num_heads: int
    kv_lora_rank: int
    rope_dim: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray      # int32 [B]
    block_table: np.ndarray   # int32 [B, max_blocks]
    q: np.ndarray             # uint16 [B, H, kv_lora_rank + rope_dim]
    pool: np.ndarray          # uint16 [nb, bs, kv_lora_rank + rope_dim]
    scale: float

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def kv_bytes(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum()) * (self.kv_lora_rank + self.rope_dim) * 2


def make_mla_batch(name, seed, seq_lens, num_heads, kv_lora_rank=512, rope_dim=64,
                   block_size=64, num_blocks=None, scale=None, with_pool=True) -> MLABatch:
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    table, nb = _assign_blocks(rng, seq_lens, block_size, num_blocks)
    dk = kv_lora_rank + rope_dim
    pool = randn_bf16(rng, (nb, block_size, dk)) if with_pool else None
    rng = np.random.default_rng([seed, 1])
    q = randn_bf16(rng, (seq_lens.shape[0], num_heads, dk))
    if scale is None:
        scale = 1.0 / math.sqrt(128 + rope_dim)
    return MLABatch(name, seed, num_heads, kv_lora_rank, rope_dim, block_size, nb,
                    seq_lens, table, q, pool, float(scale))


def mla_new_tokens(m: "MLABatch", seed_offset: int = 2):
    """The decode step's new latent entries of an MLA batch: for each request
    the token at position seq_len - 1, with kv_c [B, kv_lora_rank] and k_pe
    [B, rope_dim] drawn as N(0, 1) bf16 bits from default_rng([seed, 2]) and
    slot = block_table[i][pos // bs] * bs + pos % bs (requests of length 0
    get slot -1)."""
    rng = np.random.default_rng([m.seed, seed_offset])
    B = m.batch
    kv_c = randn_bf16(rng, (B, m.kv_lora_rank))
    k_pe = randn_bf16(rng, (B, m.rope_dim))
    slots = np.full(B, -1, np.int64)
    for i in range(B):
        n = int(m.seq_lens[i])
        if n > 0:
            pos = n - 1
            slots[i] = int(m.block_table[i, pos // m.block_size]) * m.block_size + pos % m.block_size
    return kv_c, k_pe, slots


@dataclass
class MLAPrefillBatch:
    """One prefill step of the MLA workload in the multi-head formulation:
    latent pool [nb, bs, R + dr], per-head queries [T, H, dn + dr], the
    kv_b_proj weight [H, dn + dv, R], and the step's new latent rows."""
    name: str
    seed: int
    num_heads: int
    kv_lora_rank: int
    rope_dim: int
    qk_nope_dim: int
    v_dim: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray          # int32 [N]
    query_lens: np.ndarray        # int32 [N]
    query_start_loc: np.ndarray   # int32 [N + 1]
    block_table: np.ndarray       # int32 [N, max_blocks], -1 past the end
    slot_mapping: np.ndarray      # int64 [T]
    q: np.ndarray                 # uint16 [T, H, dn + dr]
    kv_c: np.ndarray              # uint16 [T, R]  (new latent rows)
    k_pe: np.ndarray              # uint16 [T, dr]
    w_kv_b: np.ndarray            # uint16 [H, dn + dv, R]
    pool: np.ndarray              # uint16 [nb, bs, R + dr] BEFORE the write
    scale: float

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    def causal_flops(self) -> int:
        """2 * (dn + dr + dv) * H * sum_i(qlen_i * ctx_i + qlen_i (qlen_i + 1) / 2)."""
        ql = self.query_lens.astype(np.int64)
        ctx = self.seq_lens.astype(np.int64) - ql
        pairs = int((ql * ctx + ql * (ql + 1) // 2).sum())
        return 2 * (self.qk_nope_dim + self.rope_dim + self.v_dim) * self.num_heads * pairs

    def expand_flops(self) -> int:
        """2 * R * H * (dn + dv) per context token (the kv_b_proj expansion)."""
        return (2 * self.kv_lora_rank * self.num_heads * (self.qk_nope_dim + self.v_dim) *
                int(self.seq_lens.astype(np.int64).sum()))


def make_mla_prefill_batch(name, seed, seq_lens, query_lens, num_heads, kv_lora_rank=512,
                           rope_dim=64, qk_nope_dim=128, v_dim=128, block_size=64,
                           with_pool=True, scale=None) -> MLAPrefillBatch:
    """Latent pool and queries N(0, 1) bf16; kv_b_proj weight N(0, 1/R) bf16
    (so the expanded keys and values are of unit scale); new tokens are the
    last query_lens[i] positions of each request, their slots as in
    make_paged_batch."""
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int32)
    query_lens = np.asarray(query_lens, np.int32)
    assert np.all(query_lens <= seq_lens) and np.all(query_lens >= 0)
    N = seq_lens.shape[0]
    qsl = np.zeros(N + 1, np.int32)
    qsl[1:] = np.cumsum(query_lens)
    table, nb = _assign_blocks(rng, seq_lens, block_size)
    T = int(qsl[-1])
    slots = np.empty(T, np.int64)
    for i in range(N):
        ctx = int(seq_lens[i] - query_lens[i])
        for j in range(int(query_lens[i])):
            pos = ctx + j
            slots[qsl[i] + j] = int(table[i, pos // block_size]) * block_size + pos % block_size
    width = kv_lora_rank + rope_dim
    pool = randn_bf16(rng, (nb, block_size, width)) if with_pool else None
    rng = np.random.default_rng([seed, 1])
    q = randn_bf16(rng, (T, num_heads, qk_nope_dim + rope_dim))
    kv_c = randn_bf16(rng, (T, kv_lora_rank))
    k_pe = randn_bf16(rng, (T, rope_dim))
    wr = np.random.default_rng([seed, 3])
    w = (wr.standard_normal((num_heads, qk_nope_dim + v_dim, kv_lora_rank), dtype=np.float32) /
         np.float32(math.sqrt(kv_lora_rank)))
    w_kv_b = f32_to_bf16_bits(w)
    if scale is None:
        scale = 1.0 / math.sqrt(qk_nope_dim + rope_dim)
    return MLAPrefillBatch(name, seed, num_heads, kv_lora_rank, rope_dim, qk_nope_dim, v_dim,
                           block_size, nb, seq_lens, query_lens, qsl, table, slots, q, kv_c,
                           k_pe, w_kv_b, pool, float(scale))


def mla_prefill(seed: int = 7, num_seqs: int = 8, qlo: int = 256, qhi: int = 2048,
                clo: int = 0, chi: int = 4096, **kw) -> MLAPrefillBatch:
    """DeepSeek-V3 MLA chunked prefill: 8 requests, new tokens U[256, 2048],
    cached prefix U[0, 4096], 128 heads, latent 512 + rope 64, q/k nope 128,
    v 128, block size 64, scale 1/sqrt(192)."""
    rng = np.random.default_rng(seed + 1000)
    ql = rng.integers(qlo, qhi, size=num_seqs, endpoint=True).astype(np.int32)
    ctx = rng.integers(clo, chi, size=num_seqs, endpoint=True).astype(np.int32)
    return make_mla_prefill_batch(f"mla_prefill_{num_seqs}req_128h", seed, ctx + ql, ql, 128,
                                  **kw)


def make_shared_prefix_batch(name, seed, prefix_blocks, suffix_lens, query_lens, num_q_heads,
                             num_kv_heads, head_size, block_size, scale=None,
                             with_pool=True) -> PagedBatch:
    """A batch whose requests all begin with the same ``prefix_blocks`` blocks
    (the same block ids in every table row: a shared system prompt) followed
    by their own ``suffix_lens[i]`` tokens, the last ``query_lens[i]`` of which
    are the step's new tokens.  Block ids: a seeded permutation, the first
    ``prefix_blocks`` of it for the prefix, the rest handed out in request
    order.  Values as in make_paged_batch."""
    rng = np.random.default_rng(seed)
    suffix_lens = np.asarray(suffix_lens, np.int32)
    query_lens = np.asarray(query_lens, np.int32)
    assert np.all(query_lens <= suffix_lens) and np.all(query_lens >= 0)
    N = suffix_lens.shape[0]
    seq_lens = (suffix_lens + prefix_blocks * block_size).astype(np.int32)
    need = [(int(x) + block_size - 1) // block_size for x in suffix_lens]
    nb = prefix_blocks + sum(need)
    perm = rng.permutation(nb).astype(np.int32)
    max_blocks = max(1, prefix_blocks + (max(need) if need else 0))
    table = np.full((N, max_blocks), -1, np.int32)
    k = prefix_blocks
    for i, n in enumerate(need):
        table[i, :prefix_blocks] = perm[:prefix_blocks]
        table[i, prefix_blocks:prefix_blocks + n] = perm[k:k + n]
        k += n
    qsl = np.zeros(N + 1, np.int32)
    qsl[1:] = np.cumsum(query_lens)
    T = int(qsl[-1])
    slots = np.empty(T, np.int64)
    for i in range(N):
        ctx = int(seq_lens[i] - query_lens[i])
        for j in range(int(query_lens[i])):
            pos = ctx + j
            slots[qsl[i] + j] = int(table[i, pos // block_size]) * block_size + pos % block_size
    pool = randn_bf16(rng, (nb, 2, block_size, num_kv_heads, head_size)) if with_pool else None
    rng = np.random.default_rng([seed, 1])
    q = randn_bf16(rng, (T, num_q_heads, head_size))
    key = randn_bf16(rng, (T, num_kv_heads, head_size))
    value = randn_bf16(rng, (T, num_kv_heads, head_size))
    if scale is None:
        scale = 1.0 / math.sqrt(head_size)
    return PagedBatch(name, seed, num_q_heads, num_kv_heads, head_size, block_size, nb, seq_lens,
                      query_lens, qsl, table, slots, q, key, value, pool, float(scale), True)


def shared_prefix_decode(seed: int = 6, num_seqs: int = 64, prefix_tokens: int = 4096,
                         lo: int = 64, hi: int = 1024, **kw) -> PagedBatch:
    """64 decode requests (one new token each) sharing a 4096-token prompt,
    each with its own U[64, 1024] tokens after it; 32 q / 8 kv heads, d 128,
    block size 16."""
    rng = np.random.default_rng(seed + 1000)
    suf = rng.integers(lo, hi, size=num_seqs, endpoint=True).astype(np.int32)
    return make_shared_prefix_batch(f"shared_prefix_decode_{num_seqs}req_p{prefix_tokens}",
                                    seed, prefix_tokens // 16, suf, np.ones(num_seqs, np.int32),
                                    32, 8, 128, 16, **kw)


# ---------------------------------------------------------------------------
# fp8 (e4m3) KV cache inputs.
# ---------------------------------------------------------------------------

# Per-layer scales of the fp8 workloads: an fp8 K entry with code c stands for
# e4m3(c) * FP8_K_SCALE, a V entry for e4m3(c) * FP8_V_SCALE.  Neither is a
# power of two, so quantising a new key (x / scale) rounds.
FP8_K_SCALE = float(np.float32(0.0153))
FP8_V_SCALE = float(np.float32(0.0211))


def e4m3_codes(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """Uniformly random finite e4m3 codes as uint8: each of the 254 codes other
    than the two NaN codes (0x7F, 0xFF) is equally likely.  Chunked as
    randn_bf16."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint8)

    def fill(gen, a, m):
        r = gen.integers(0, 254, size=m, dtype=np.uint8)
        r[r >= 0x7F] += 1
        out[a:a + m] = r

    _chunked_fill(rng, n, chunk, fill)
    return out.reshape(shape)


def fp8_pool(b: "PagedBatch") -> np.ndarray:
    """An fp8 pool with the shape of ``b``'s pool, [nb, 2, bs, Hkv, d] uint8,
    filled with random finite codes drawn from ``default_rng([seed, 2])``."""
    rng = np.random.default_rng([b.seed, 2])
    return e4m3_codes(rng, (b.num_blocks, 2, b.block_size, b.num_kv_heads, b.head_size))


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def tiny_paged(seed: int = 1) -> PagedBatch:
    """3 requests, seq_lens {5, 17, 40}, query_lens {5, 1, 1}, 4 q / 2 kv heads,
    head_size 64, block_size 16, a 16-block pool, scale 1/8, causal."""
    return make_paged_batch("tiny_paged_3req_d64", seed, [5, 17, 40], [5, 1, 1], 4, 2, 64,
                            16, num_blocks=16, scale=1.0 / 8.0)


def gqa_decode(seed: int = 2, num_seqs: int = 64, lo: int = 128, hi: int = 4096,
               **kw) -> PagedBatch:
    """Llama-3-8B attention shape: 64 requests x 1 query, seq_lens U[128, 4096],
    32 q / 8 kv heads, head_size 128, block_size 16."""
    rng = np.random.default_rng(seed + 1000)
    seq = rng.integers(lo, hi, size=num_seqs, endpoint=True).astype(np.int32)
    return make_paged_batch(f"gqa_decode_{num_seqs}req_seq{lo}-{hi}_32q8kv_d128", seed, seq,
                            np.ones(num_seqs, np.int32), 32, 8, 128, 16, **kw)


def chunked_prefill(seed: int = 3, num_seqs: int = 16, qlo: int = 256, qhi: int = 2048,
                    clo: int = 0, chi: int = 4096, **kw) -> PagedBatch:
    """16 requests, new-query lengths U[256, 2048], cached prefix U[0, 4096],
    32 q / 8 kv heads, head_size 128, block_size 16, causal."""
    rng = np.random.default_rng(seed + 1000)
    ql = rng.integers(qlo, qhi, size=num_seqs, endpoint=True).astype(np.int32)
    ctx = rng.integers(clo, chi, size=num_seqs, endpoint=True).astype(np.int32)
    return make_paged_batch(f"chunked_prefill_{num_seqs}req_32q8kv_d128", seed, ctx + ql, ql,
                            32, 8, 128, 16, **kw)


def long_decode(seed: int = 4, num_seqs: int = 8, seq_len: int = 131072, **kw) -> PagedBatch:
    """Llama-3-70B attention shape: 8 requests x 1 query at seq_len 131072,
    64 q / 8 kv heads, head_size 128, block_size 16."""
    return make_paged_batch(f"long_decode_{num_seqs}x{seq_len}_64q8kv_d128", seed,
                            np.full(num_seqs, seq_len, np.int32), np.ones(num_seqs, np.int32),
                            64, 8, 128, 16, **kw)


def mla_decode(seed: int = 5, batch: int = 128, lo: int = 1024, hi: int = 8192,
               **kw) -> MLABatch:
    """DeepSeek-V3 shape: 128 requests x 1 query, 128 heads over one 576-wide
    latent KV head (kv_c 512 | k_pe 64), value = first 512, seq_lens
    U[1024, 8192], block_size 64, scale 1/sqrt(192)."""
    rng = np.random.default_rng(seed + 1000)
    seq = rng.integers(lo, hi, size=batch, endpoint=True).astype(np.int32)
    return make_mla_batch(f"mla_decode_{batch}req_128h_576", seed, seq, 128, 512, 64, 64,
                          scale=1.0 / math.sqrt(192.0), **kw)

