/*
 * pa.h -- C ABI of the GB300 paged-attention library (libpa.so).
 *
 * The library implements the hot path that every paged-attention backend
 * wraps, as the two-step kernel contract of "Attention Backends" (vLLM
 * model-execution notes), section "What 'paged attention' requires of a
 * kernel", states it: (1) write the step's new keys and values into the cache
 * at slot_mapping; (2) for each request, attend from its queries over its
 * first seq_len tokens, fetched block by block through its block_table row.
 * Split-KV decode and the LSE merge follow "Chapter 1: attention backends"
 * (zero-to-sglang), section 3.1, and the data-flow section of "Triton and
 * MLA" (vllm-arch-zh); MLA latent decode follows the latter.
 *
 * Conventions for every entry point:
 *  - Every data pointer is a DEVICE pointer owned by the caller; the library
 *    allocates nothing and never synchronises the host.  Its only state is a
 *    cached SM count and tensor-map encoder per device, the device error word,
 *    and the fixed 16 MiB device array of pa_decode_noalloc (present on every
 *    device that loads the library, used only by that entry point).
 *  - bf16 tensors are passed as `const void*` / `void*` and hold IEEE
 *    bfloat16 values; every tensor is dense and row-major (C order) with the
 *    shape stated below.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously on it.
 *  - Arguments are validated on the host before anything is launched; a call
 *    that returns anything but PA_OK has launched nothing (PA_ERR_CUDA: the
 *    launch itself failed).
 *  - Index types: block_table, query_start_loc and seq_lens are int32;
 *    slot_mapping is int64.
 *  - The standard KV pool is [num_blocks, 2, block_size, num_kv_heads,
 *    head_size] (index 0 = keys, 1 = values), the layout "AttentionBackend:
 *    attention backend abstraction layer" (vllm-arch-zh), design-motivation
 *    list, gives for FlashAttention.  The MLA pool is [num_blocks, block_size,
 *    kv_lora_rank + rope_dim] (same page; "Triton and MLA", design list).
 *  - Block ids in block_table are checked on the device against num_blocks:
 *    an id outside [0, num_blocks) is never dereferenced; its tokens are
 *    treated as masked and PA_DEVERR_BLOCK_ID is recorded in the device error
 *    word (read it with pa_get_device_error).  Entries past
 *    ceil(seq_len / block_size) are never read.
 *  - LSE outputs are fp32 natural-log (log-sum-exp of scale * q.k), matching
 *    the "lse_base_on_e" convention of the abstraction-layer page.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID = 1,     /* bad argument: null pointer, size, divisibility */
  PA_ERR_UNSUPPORTED = 2, /* valid on the pages but not built here (head size, width) */
  PA_ERR_CUDA = 3         /* a CUDA launch or query failed */
} pa_status;

/* Device error word bits (pa_get_device_error). */
#define PA_DEVERR_BLOCK_ID 1  /* a block_table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT 2      /* a slot_mapping entry >= num_blocks * block_size */
#define PA_DEVERR_TIMEOUT 4   /* a kernel gave up a bounded wait; its outputs are invalid */
#define PA_DEVERR_LENGTH 8    /* a request's lengths break a call's stated precondition */

/* Shape of a standard-layout paged batch. */
typedef struct pa_shape {
  int num_seqs;           /* N: requests in the batch                          */
  int num_q_heads;        /* Hq                                                 */
  int num_kv_heads;       /* Hkv; Hq % Hkv == 0, q head h reads kv head h/(Hq/Hkv) */
  int head_size;          /* d                                                  */
  int block_size;         /* tokens per cache block; a positive multiple of 16  */
  int num_blocks;         /* blocks in the pool; at least 1                     */
  int max_blocks_per_seq; /* columns of block_table; at least 1                 */
} pa_shape;

/*
 * Step 1 of the kernel contract: the cache write.
 *   For t < num_tokens with slot = slot_mapping[t] >= 0:
 *     kv_cache[slot / bs, 0, slot % bs, :, :] = key[t, :, :]
 *     kv_cache[slot / bs, 1, slot % bs, :, :] = value[t, :, :]
 *   A bit copy.  slot < 0 skips the token.  A slot >= num_blocks * bs is not
 *   written and sets PA_DEVERR_SLOT.
 * key, value: [num_tokens, Hkv, d] bf16.  kv_cache: standard pool, in-out.
 * Uses shape->num_kv_heads, head_size (a multiple of 8), block_size,
 * num_blocks.  num_tokens == 0 is a no-op.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* kv_cache,
                               const int64_t* slot_mapping, int num_tokens,
                               const pa_shape* shape, void* stream);

/*
 * Step 2 of the kernel contract: varlen paged attention (prefill, chunked
 * prefill, mixed batches).  For request i, rows j in
 * [query_start_loc[i], query_start_loc[i+1]) are its qlen_i newest tokens:
 * row j sits at position p_j = seq_lens[i] - qlen_i + (j - query_start_loc[i]).
 * For q head h (kv head h / (Hq/Hkv)):
 *   out[j, h, :] = softmax(scale * q[j, h, :] . K[p, :] for visible p) . V
 *   lse[j, h]    = ln sum_p exp(scale * q[j, h, :] . K[p, :])
 * where p is visible if p <= p_j (causal != 0) or p < seq_lens[i] (causal == 0);
 * O = softmax(Q K^T / sqrt(d_h) + M) V of "Chapter 1: attention backends",
 * section 2.1, with the mask M.
 * q, out: [total_q, Hq, d] bf16.  lse: [total_q, Hq] fp32, nullable.
 * query_start_loc: [N + 1], non-decreasing, query_start_loc[N] == total_q.
 * seq_lens: [N] with seq_lens[i] >= qlen_i.  max_query_len >= every qlen_i
 * (sizes the grid; rows beyond it are not computed).
 * Supported: head_size in {64, 128}.  A row with nothing visible gets o = 0
 * and lse = -inf.  total_q == 0 is a no-op.
 */
pa_status pa_varlen_fwd(const void* q, const void* kv_cache, const int32_t* block_table,
                        const int32_t* query_start_loc, const int32_t* seq_lens,
                        int total_q, int max_query_len, const pa_shape* shape,
                        float scale, int causal, void* out, float* lse, void* stream);

/*
 * Varlen paged attention with a sliding window: pa_varlen_fwd with causal
 * masking in which row j at position p_j sees only the sliding_window newest
 * positions up to its own, p_j - sliding_window < p <= p_j.  The pages name
 * sliding_window only as an input of backend selection ("attention-backend-
 * selection", trigger conditions); this reading (the W newest positions,
 * the row's own included) is the library's.  sliding_window >= 1 (else
 * PA_ERR_INVALID); a window at least as long as every sequence equals
 * pa_varlen_fwd with causal = 1.  Other arguments as for pa_varlen_fwd.
 */
pa_status pa_varlen_fwd_window(const void* q, const void* kv_cache, const int32_t* block_table,
                               const int32_t* query_start_loc, const int32_t* seq_lens,
                               int total_q, int max_query_len, const pa_shape* shape, float scale,
                               int sliding_window, void* out, float* lse, void* stream);

/*
 * Cascade (shared-prefix) attention ("Attention Backends", section "Cascade
 * attention": when every running request shares its first
 * num_common_prefix_blocks blocks, the shared part is processed once and the
 * per-request parts separately).  The result is that of pa_varlen_fwd on the
 * same arguments; it is computed as
 *   pass 1: every query row of the batch against the first
 *           P = num_common_prefix_blocks * block_size tokens, read once per kv
 *           head through row 0 of block_table, without a mask, cut into
 *           num_prefix_splits pieces of whole 128-token tiles -> workspace
 *           slots [0, num_prefix_splits);
 *   pass 2: request i against its own tokens from position P on (table
 *           columns from num_common_prefix_blocks), with the call's mask, cut
 *           into num_suffix_splits pieces as pa_decode_splitkv cuts a batch
 *           whose longest sequence is max_seq_len - P -> slots
 *           [num_prefix_splits, num_prefix_splits + num_suffix_splits).  A
 *           batch of one query per request (total_q == num_seqs,
 *           max_query_len == 1) runs this pass on the split-KV decode kernel;
 *   merge:  the pa_lse_merge of all the slots -> out, lse.
 * Preconditions: the first num_common_prefix_blocks entries of every table
 * row are the same block ids; with causal != 0 every query lies after the
 * prefix (seq_lens[i] - qlen_i >= P; a request that breaks it sets
 * PA_DEVERR_LENGTH and its rows are invalid).  max_seq_len >= every
 * seq_lens[i] (sizes the suffix pieces; a smaller value costs speed, never
 * correctness).
 * workspace: pa_decode_workspace_bytes(total_q, Hq, num_prefix_splits +
 * num_suffix_splits, d) bytes (fp32 [total_q, Hq, slots, d + 1]).
 * num_common_prefix_blocks == 0 runs pa_varlen_fwd (workspace untouched).
 * Other arguments as for pa_varlen_fwd; head_size in {64, 128}, Hq / Hkv <= 16.
 */
pa_status pa_cascade_fwd(const void* q, const void* kv_cache, const int32_t* block_table,
                         const int32_t* query_start_loc, const int32_t* seq_lens, int total_q,
                         int max_query_len, int max_seq_len, int num_common_prefix_blocks,
                         int num_prefix_splits, int num_suffix_splits, const pa_shape* shape,
                         float scale, int causal, float* workspace, void* out, float* lse,
                         void* stream);

/*
 * A num_prefix_splits for pa_cascade_fwd: enough pieces of the prefix that
 * pass 1 has one unit (256 packed query rows x kv head x piece) per SM, at
 * most one per 128 prefix tokens, at least 1.  sm_count <= 0 means the
 * current device's.
 */
int pa_cascade_prefix_splits(int total_q, int num_q_heads, int num_kv_heads, int prefix_tokens,
                             int sm_count);

/*
 * Split-count rule of "Triton and MLA", key-files list (_compute_num_kv_splits):
 * min(ceil(max_seq_len / 512), 2 * sm_count), at least 1.  sm_count <= 0
 * means the current device's SM count.
 */
int pa_num_kv_splits(int max_seq_len, int sm_count);

/*
 * Bytes of the split-KV workspace [num_seqs, num_q_heads, num_splits, dv + 1]
 * fp32: each split's normalised partial output followed by its LSE ("the +1
 * stores the LSE", data-flow section of "Triton and MLA").  0 on bad sizes.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_splits, int dv);

/*
 * Split-KV decode, stage 1 (one query per request; the query attends over
 * all seq_lens[i] cached tokens).  The split count S is derived from the
 * batch's longest sequence ("Triton and MLA", key files), so the sequence
 * axis is cut the same way for every request: with
 *   C = bs * ceil(ceil(max_seq_len / S) / bs),
 * split s of request i covers the tokens [s*C, min((s+1)*C, seq_i)), and the
 * last split (s = S-1) runs to seq_i (so a max_seq_len below the true maximum
 * costs speed, never correctness).  For each q head h it writes the split's
 * softmax-normalised output and natural-log LSE:
 *   workspace[i, h, s, 0:d] = o_s,  workspace[i, h, s, d] = lse_s
 * An empty split writes o_s = 0, lse_s = -inf.
 * q: [N, Hq, d] bf16.  workspace: pa_decode_workspace_bytes(N, Hq, S, d) bytes.
 * max_seq_len >= 0: the batch's longest seq_len (sizes C).
 * Supported: head_size in {64, 128}, Hq / Hkv <= 16.
 */
pa_status pa_decode_splitkv(const void* q, const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, const pa_shape* shape, float scale,
                            int num_splits, int max_seq_len, float* workspace, void* stream);

/*
 * Split-KV stage 2: merge S partials per (request, head) by their LSE:
 *   M = max_s lse_s,  w_s = exp(lse_s - M),
 *   out = sum_s w_s o_s / sum_s w_s  (rounded to bf16),  lse = M + ln sum_s w_s.
 * All partials empty: out = 0, lse = -inf.
 * workspace: [num_seqs, num_q_heads, num_splits, dv + 1] fp32.
 * out: [num_seqs, num_q_heads, dv] bf16.  lse: [num_seqs, num_q_heads], nullable.
 */
pa_status pa_lse_merge(const float* workspace, int num_seqs, int num_q_heads,
                       int num_splits, int dv, void* out, float* lse, void* stream);

/*
 * MLA latent decode ("Triton and MLA", data flow: forward_mqa): MQA over a
 * single latent KV head.  For request b and head h:
 *   s_p = scale * q[b, h, :] . c[p, :]   (all kv_lora_rank + rope_dim entries)
 *   out[b, h, :] = softmax(s) . c[:, 0:kv_lora_rank],  lse[b, h] = ln sum exp(s_p)
 * where c[p] = kv_cache[block_table[b][p / bs], p % bs, :], p < seq_lens[b].
 * q: [batch, num_heads, kv_lora_rank + rope_dim] bf16 (q_nope absorbed | q_pe).
 * kv_cache: [num_blocks, block_size, kv_lora_rank + rope_dim] bf16.
 * out: [batch, num_heads, kv_lora_rank] bf16.  lse: [batch, num_heads] fp32, nullable.
 * The call runs split-KV stage 1 into `workspace`
 * (pa_decode_workspace_bytes(batch, num_heads, num_splits, kv_lora_rank) bytes,
 * splits cut as for pa_decode_splitkv from max_seq_len) and then the LSE merge;
 * with num_splits == 1 and `out` 16-byte aligned it writes out and lse
 * directly and leaves the workspace untouched (it must still be passed).
 * Supported: kv_lora_rank == 512, rope_dim == 64, num_heads a multiple of 64,
 * block_size a multiple of 32.  num_blocks and max_blocks_per_seq must be at
 * least 1 (a pool with no blocks is PA_ERR_INVALID, even for a batch whose
 * requests are all empty).
 */
pa_status pa_mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                        const int32_t* seq_lens, int batch, int num_heads, int kv_lora_rank,
                        int rope_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                        int max_seq_len, float scale, int num_splits, float* workspace, void* out,
                        float* lse, void* stream);

/*
 * A num_splits for pa_decode_splitkv / pa_decode_splitkv_fp8 chosen from the
 * batch as well as max_seq_len and the SM count (the library's planner; the
 * page's rule is pa_num_kv_splits).  Every (request, kv head, split) is one
 * CTA, and each CTA pays a fixed start-up and combine cost, so the planner
 * takes just enough splits for about twelve CTAs per SM, never more than
 * the page's rule gives:
 *   S = min(max(1, ceil(12 * sm_count / (num_seqs * num_kv_heads))),
 *           pa_num_kv_splits(max_seq_len, sm_count)).
 * sm_count <= 0 means the current device's SM count; num_seqs <= 0 or
 * num_kv_heads <= 0 gives 1.
 */
int pa_decode_num_kv_splits(int num_seqs, int num_kv_heads, int max_seq_len, int sm_count);

/*
 * A num_splits for pa_mla_decode, chosen from the batch, the head count, the
 * longest sequence and the SM count (the split count of "Triton and MLA",
 * key-files list, _compute_num_kv_splits, is likewise chosen from max_seq_len
 * and sm_count; this rule is the library's for the MLA kernel).  One
 * (split, request, group of 128 heads) unit runs on a pair of SMs, and each
 * split adds a [128, kv_lora_rank + 1] fp32 partial per request and head
 * group (written once and read once by the merge: ~456 tokens' worth of
 * cache bytes), so the rule takes just enough splits to give every SM pair
 * one unit, and never splits finer than the page's 512-token pieces:
 *   units = batch * ceil(num_heads / 128),
 *   S = min(ceil((sm_count / 2) / units), ceil(max_seq_len / 512)), at least 1.
 * sm_count <= 0 means the current device's SM count; batch <= 0 or
 * num_heads <= 0 gives 1.
 */
int pa_mla_num_kv_splits(int batch, int num_heads, int max_seq_len, int sm_count);

/*
 * fp8 KV cache.  The pool holds e4m3 codes (OCP FP8 "fn": 1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; largest finite 448; 0x7F / 0xFF NaN),
 * one byte per element, in the standard layout [num_blocks, 2, block_size,
 * num_kv_heads, head_size].  A K entry with code c stands for
 * e4m3(c) * k_scale and a V entry for e4m3(c) * v_scale: the per-layer
 * scales that the decode kernel always receives ("Triton and MLA", data flow,
 * decode_attention_fwd's k_scale / v_scale).  Both scales must be finite
 * and > 0 (else PA_ERR_INVALID).
 */

/*
 * Step 1 with an fp8 pool: the quantising cache write.
 *   For t < num_tokens with slot = slot_mapping[t] >= 0 and every (h, e):
 *     kv_cache[slot / bs, 0, slot % bs, h, e] = E(key[t, h, e] / k_scale)
 *     kv_cache[slot / bs, 1, slot % bs, h, e] = E(value[t, h, e] / v_scale)
 *   where the quotient is the fp32 IEEE quotient of the bf16 value (widened
 *   exactly) by the scale, and E is the e4m3 code nearest to it, ties to
 *   even, magnitudes beyond 448 (infinities included) saturating to +-448;
 *   NaN gives a NaN code.  Reading the write side as the inverse of the read
 *   side is this library's reading; the pages state only the read side.
 *   slot < 0 skips the token; a slot >= num_blocks * bs is not written and
 *   sets PA_DEVERR_SLOT.
 * key, value: [num_tokens, Hkv, d] bf16, 16-byte aligned.  kv_cache: fp8
 * pool (bytes), 16-byte aligned, in-out.  Uses shape->num_kv_heads,
 * head_size (a multiple of 16), block_size, num_blocks.  num_tokens == 0 is a
 * no-op.
 */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* kv_cache,
                                   const int64_t* slot_mapping, int num_tokens,
                                   const pa_shape* shape, float k_scale, float v_scale,
                                   void* stream);

/*
 * Split-KV decode, stage 1, over an fp8 pool: pa_decode_splitkv with every
 * K entry read as e4m3(c) * k_scale and every V entry as e4m3(c) * v_scale
 * (same splits, same workspace layout and contents; merge with
 * pa_lse_merge).  The products are taken on f16 tensor-core operands: the
 * codes convert to f16 exactly, q is rounded bf16 -> f16 (exact for |q| in
 * [2^-14, 65504]; larger magnitudes are not supported), and the softmax
 * weights are rounded to f16; accumulation is fp32.
 * q: [N, Hq, d] bf16, 4-byte aligned.  kv_cache: fp8 pool, 16-byte aligned.
 * Supported: head_size in {64, 128}, Hq / Hkv <= 16.
 */
pa_status pa_decode_splitkv_fp8(const void* q, const void* kv_cache, const int32_t* block_table,
                                const int32_t* seq_lens, const pa_shape* shape, float scale,
                                float k_scale, float v_scale, int num_splits, int max_seq_len,
                                float* workspace, void* stream);

/*
 * The MLA cache write, the step before pa_mla_decode ("Triton and MLA": the
 * cache stores one vector per token, the compressed latent kv_c followed by
 * the rotary key part k_pe; its shape is (num_blocks, block_size, head_size)).
 *   For t < num_tokens with slot = slot_mapping[t] >= 0:
 *     kv_cache[slot / bs, slot % bs, 0:kv_lora_rank] = kv_c[t, :]
 *     kv_cache[slot / bs, slot % bs, kv_lora_rank:]  = k_pe[t, :]
 *   A bit copy.  slot < 0 skips the token; a slot >= num_blocks * bs is not
 *   written and sets PA_DEVERR_SLOT.
 * kv_c: [num_tokens, kv_lora_rank] bf16; k_pe: [num_tokens, rope_dim] bf16;
 * kv_cache: [num_blocks, block_size, kv_lora_rank + rope_dim] bf16, in-out.
 * All 16-byte aligned.  Supported: kv_lora_rank and rope_dim multiples of 8.
 */
pa_status pa_mla_cache_write(const void* kv_c, const void* k_pe, void* kv_cache,
                             const int64_t* slot_mapping, int num_tokens, int kv_lora_rank,
                             int rope_dim, int block_size, int num_blocks, void* stream);

/*
 * MLA prefill, multi-head formulation ("Attention Backends", section "Latent
 * attention is a different cache, not just a different kernel": prefill and
 * decode use different formulations of the same mathematics;
 * "AttentionBackend: attention backend abstraction layer": forward_mha).
 * Widths are DeepSeek-V3's: kv_lora_rank 512, rope_dim 64, qk_nope 128,
 * v 128 (the cache row is 576 wide, the query 192, the output 128).
 *
 * pa_mla_expand_kv -- step 1: for every request i and context token
 * t < seq_lens[i], with c = kv_cache[block_table[i][t / bs]][t % bs]:
 *   k_ws[i][t][h][0:128]   = bf16(w_kv_b[h][0:128] . c[0:512])
 *   k_ws[i][t][h][128:192] = c[512:576]                       (k_pe)
 *   v_ws[i][t][h][0:128]   = bf16(w_kv_b[h][128:256] . c[0:512])
 * fp32 accumulation, round to nearest even; entries for t >= seq_lens[i] are
 * not written.  w_kv_b: the model's kv_b_proj weight [num_heads][256][512]
 * bf16.  k_ws: [num_seqs][max_seq_len][num_heads][192] bf16, v_ws:
 * [num_seqs][max_seq_len][num_heads][128] bf16 (together
 * pa_mla_prefill_workspace_bytes bytes).  max_seq_len >= every seq_lens[i]
 * (a shorter one is the caller's error: tokens past it are not expanded).
 * A block id outside [0, num_blocks) sets PA_DEVERR_BLOCK_ID and its tokens
 * expand as zero latents.  k_ws and v_ws 32-byte aligned (rows are written
 * with 32-byte stores), the other pointers 16-byte aligned.
 */
size_t pa_mla_prefill_workspace_bytes(int num_seqs, int max_seq_len, int num_heads);
pa_status pa_mla_expand_kv(const void* kv_cache, const void* w_kv_b, const int32_t* block_table,
                           const int32_t* seq_lens, int num_seqs, int num_heads, int block_size,
                           int num_blocks, int max_blocks_per_seq, int max_seq_len, void* k_ws,
                           void* v_ws, void* stream);

/*
 * pa_mla_prefill -- the whole forward_mha step: pa_mla_expand_kv into the
 * workspace (k_ws first, then v_ws, together pa_mla_prefill_workspace_bytes(
 * num_seqs, max_seq_len, num_heads) bytes), then varlen attention with
 * per-head keys [k_nope | k_pe] (192) and values v (128):
 *   out[j, h, :] = softmax(scale * q[j, h, :] . K_h[p] for visible p) . V_h
 *   lse[j, h]    = ln sum_p exp(scale * q[j, h, :] . K_h[p])
 * with visibility as in pa_varlen_fwd (causal: bottom-right aligned).
 * q: [total_q, num_heads, 192] bf16 ([q_nope | q_pe]); out: [total_q,
 * num_heads, 128] bf16; lse: [total_q, num_heads] fp32, nullable.
 * query_start_loc, seq_lens, max_query_len as for pa_varlen_fwd; the new
 * tokens must already be in kv_cache (pa_mla_cache_write).  workspace
 * 32-byte aligned; q, kv_cache, w_kv_b and out 16-byte aligned.
 */
pa_status pa_mla_prefill(const void* q, const void* kv_cache, const void* w_kv_b,
                         const int32_t* block_table, const int32_t* query_start_loc,
                         const int32_t* seq_lens, int total_q, int max_query_len, int num_seqs,
                         int num_heads, int block_size, int num_blocks, int max_blocks_per_seq,
                         int max_seq_len, float scale, int causal, void* workspace, void* out,
                         float* lse, void* stream);

/* Size of the fixed device array pa_decode_noalloc keeps its split partials in. */
#define PA_NOALLOC_WORKSPACE_BYTES (16u * 1024u * 1024u)

/*
 * Split-KV decode (stage 1 and the LSE merge, exactly as pa_decode_splitkv
 * followed by pa_lse_merge) that allocates nothing and takes no workspace.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory -- a host application that owns every device
 * allocation and gives the library no allocator, or a path that must never
 * call cudaMalloc -- and so cannot pass a workspace.  The split partials go
 * to a fixed device array of PA_NOALLOC_WORKSPACE_BYTES inside the library,
 * which every device that loads the library keeps until the process exits.
 *   q: [N, Hq, d] bf16;  out: [N, Hq, d] bf16;  lse: [N, Hq] fp32, nullable;
 *   max_seq_len as for pa_decode_splitkv.
 * Returns PA_ERR_INVALID if N * Hq * num_splits * (d + 1) * 4 bytes exceeds
 * PA_NOALLOC_WORKSPACE_BYTES (use fewer splits, or pa_decode_splitkv with a
 * workspace of your own).  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make it before any stream capture begins.  All calls share the array:
 * calls whose work may overlap on the GPU (unordered streams) race on it.
 */
pa_status pa_decode_noalloc(const void* q, const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, const pa_shape* shape, float scale,
                            int num_splits, int max_seq_len, void* out, float* lse,
                            void* stream);

/* Human-readable name of a status. */
const char* pa_status_string(pa_status status);

/*
 * Reads and clears the current device's error word (PA_DEVERR_* bits set by
 * earlier kernels).  Synchronises `stream` first.  *code receives the bits.
 */
pa_status pa_get_device_error(int* code, void* stream);

/* SM count of the current device (cached per device); -1 on error. */
int pa_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
