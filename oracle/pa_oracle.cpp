// Paged-attention oracle: TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU restatement of what the paged-attention hot path
// computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
// leg may load it; the product library never does, and this file shares no
// code, header or constant with the CUDA path.
//
// Sources (page title, section):
//  * "Attention Backends" (vLLM model-execution notes), section
//    "What 'paged attention' requires of a kernel": the inputs (queries,
//    new K/V, the whole cache, block_table[N, max_blocks], slot_mapping[T],
//    query_start_loc[N+1], seq_lens[N]) and the two steps: (1) write the T new
//    keys/values at slot_mapping, (2) for each request attend from its
//    queries over its first seq_len tokens, fetched through its block_table
//    row.  Section "Code": slot = block_table[pos / bs] * bs + pos % bs, and
//    paged attention equals contiguous attention exactly.
//  * "AttentionBackend: attention backend abstraction layer" (vllm-arch-zh),
//    design-motivation list: the standard pool layout
//    [num_blocks, 2, block_size, num_kv_heads, head_size] and the MLA pool
//    [num_blocks, block_size, head_size]; LSE in natural log.
//  * "Triton and MLA" (vllm-arch-zh, zh-TW), data-flow section: MLA decode is
//    MQA over one 576-wide [kv_c 512 | k_pe 64] cache vector whose first 512
//    entries are the value; split-KV partials carry their LSE in slot
//    [Dv] of a [B, H, S, Dv + 1] fp32 workspace and are merged by LSE.
//  * "Chapter 1: attention backends" (zero-to-sglang), section 2.1:
//    O = softmax(Q K^T / sqrt(d_h) + M) V; section 3.1: split-KV partials
//    merged with their softmax normalisers; section 4.1 / Fig. 5c: the
//    online-softmax merge of two blocks.
//
// Every floating-point step is done in double.  bf16 inputs are widened
// exactly (a bf16 bit pattern is the top half of an IEEE float).
//
// Readings where the pages are silent (each also listed in the design notes):
//  * causal alignment is bottom-right: the qlen_i new queries of request i are
//    its last qlen_i positions, and query row j sees positions <= its own;
//  * GQA groups are contiguous: q head h reads kv head h / (Hq / Hkv);
//  * the split count comes from the batch's longest sequence ("Triton and
//    MLA", key files), so the sequence axis is cut uniformly for the whole
//    batch: split s covers [s*C, (s+1)*C) of each request, clipped to its
//    seq_len, with C = bs * ceil(ceil(max_seq_len / S) / bs), and the last
//    split also takes any tokens past (S-1)*C; an empty split has o = 0 and
//    lse = -inf;
//  * a query with nothing visible (seq_len = 0) gives o = 0, lse = -inf;
//  * a sliding window of W positions (the pages name the parameter only, as
//    an input of backend selection) keeps the W newest positions a causal
//    row sees: row j at position p_j sees p_j - W < p <= p_j.  It is defined
//    for causal attention only.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

inline double widen(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}
inline double widen(double x) { return x; }

// Runs fn(item) for item in [0, n) on `threads` host threads.
template <typename F>
void parallel_for(int64_t n, int threads, F fn) {
  if (threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next(0);
  std::vector<std::thread> pool;
  int t = threads < n ? threads : static_cast<int>(n);
  for (int k = 0; k < t; ++k) {
    pool.emplace_back([&]() {
      for (;;) {
        int64_t i = next.fetch_add(1);
        if (i >= n) break;
        fn(i);
      }
    });
  }
  for (auto& th : pool) th.join();
}

// softmax(scale * q.K^T) V over n rows of K (width dk) and V (width dv).
// K and V are contiguous [n][dk] / [n][dv] fp64 arrays.  Writes o[dv] and
// the natural-log LSE.  n == 0 gives o = 0, lse = -inf.
void attend(const double* q, const double* K, const double* V, int64_t n,
            int dk, int dv, double scale, double* o, double* lse) {
  for (int e = 0; e < dv; ++e) o[e] = 0.0;
  if (n <= 0) {
    *lse = kNegInf;
    return;
  }
  std::vector<double> s(static_cast<size_t>(n));
  double m = kNegInf;
  for (int64_t p = 0; p < n; ++p) {
    double acc = 0.0;
    const double* k = K + p * dk;
    for (int e = 0; e < dk; ++e) acc += q[e] * k[e];
    s[p] = scale * acc;
    if (s[p] > m) m = s[p];
  }
  double l = 0.0;
  for (int64_t p = 0; p < n; ++p) {
    s[p] = std::exp(s[p] - m);
    l += s[p];
  }
  for (int64_t p = 0; p < n; ++p) {
    const double w = s[p] / l;
    const double* v = V + p * dv;
    for (int e = 0; e < dv; ++e) o[e] += w * v[e];
  }
  *lse = m + std::log(l);
}

// Gathers the first seq_len tokens of kv head g of one request from the
// standard pool [nb][2][bs][Hkv][d] into contiguous K[seq][d], V[seq][d].
// Returns false if a block id is outside [0, nb).
template <typename E>
bool gather_standard(const E* pool, const int32_t* table_row, int64_t seq_len,
                     int g, int Hkv, int d, int bs, int64_t nb,
                     std::vector<double>& K, std::vector<double>& V) {
  K.assign(static_cast<size_t>(seq_len) * d, 0.0);
  V.assign(static_cast<size_t>(seq_len) * d, 0.0);
  for (int64_t p = 0; p < seq_len; ++p) {
    const int64_t blk = table_row[p / bs];
    if (blk < 0 || blk >= nb) return false;
    const int64_t off = p % bs;
    const E* krow = pool + (((blk * 2 + 0) * bs + off) * Hkv + g) * d;
    const E* vrow = pool + (((blk * 2 + 1) * bs + off) * Hkv + g) * d;
    for (int e = 0; e < d; ++e) {
      K[p * d + e] = widen(krow[e]);
      V[p * d + e] = widen(vrow[e]);
    }
  }
  return true;
}

template <typename E>
int paged_attention(const E* q, const E* pool, const int32_t* block_table,
                    int max_blocks, const int32_t* query_start_loc,
                    const int32_t* seq_lens, int N, int Hq, int Hkv, int d,
                    int bs, int64_t nb, double scale, int causal, int window,
                    const uint8_t* row_mask, double* out, double* lse,
                    int threads) {
  if (Hkv <= 0 || Hq % Hkv != 0 || bs <= 0 || d <= 0) return -1;
  if (window < 0 || (window > 0 && !causal)) return -1;
  const int grp = Hq / Hkv;
  std::atomic<int> bad(0);
  parallel_for(static_cast<int64_t>(N) * Hkv, threads, [&](int64_t item) {
    const int i = static_cast<int>(item / Hkv);
    const int g = static_cast<int>(item % Hkv);
    const int64_t q0 = query_start_loc[i], q1 = query_start_loc[i + 1];
    const int64_t seq = seq_lens[i];
    const int64_t qlen = q1 - q0;
    if (qlen <= 0) return;
    if (qlen > seq) {
      bad = 1;
      return;
    }
    bool any = row_mask == nullptr;
    for (int64_t j = q0; j < q1 && !any; ++j) any = row_mask[j] != 0;
    if (!any) return;
    std::vector<double> K, V, qv(d);
    if (!gather_standard(pool, block_table + static_cast<int64_t>(i) * max_blocks,
                         seq, g, Hkv, d, bs, nb, K, V)) {
      bad = 1;
      return;
    }
    const int64_t ctx = seq - qlen;
    for (int64_t j = q0; j < q1; ++j) {
      if (row_mask && !row_mask[j]) continue;
      const int64_t pos = ctx + (j - q0);          // absolute position of row j
      const int64_t visible = causal ? pos + 1 : seq;
      // Sliding window: the row sees only its `window` newest positions.
      const int64_t first = (window > 0 && visible > window) ? visible - window : 0;
      for (int r = 0; r < grp; ++r) {
        const int h = g * grp + r;
        const E* qr = q + (j * Hq + h) * d;
        for (int e = 0; e < d; ++e) qv[e] = widen(qr[e]);
        attend(qv.data(), K.data() + first * d, V.data() + first * d, visible - first, d, d,
               scale, out + (j * Hq + h) * d, lse + j * Hq + h);
      }
    }
  });
  return bad ? -1 : 0;
}

// Split boundaries.  The sequence axis is cut into S pieces of
// C = bs * ceil(ceil(max_seq_len / S) / bs) tokens, the same for every
// request of the batch (max_seq_len is the value the split count is computed
// from); split s covers [s*C, (s+1)*C) clipped to the request, and the last
// split also takes everything past (S-1)*C.
inline void split_range(int64_t seq, int64_t max_seq, int S, int bs, int s,
                        int64_t* a, int64_t* b) {
  if (max_seq < 1) max_seq = 1;
  const int64_t per = (max_seq + S - 1) / S;          // ceil(max_seq / S)
  const int64_t chunk = ((per + bs - 1) / bs) * bs;   // rounded up to blocks
  *a = s * chunk;
  *b = (s == S - 1) ? seq : *a + chunk;
  if (*a > seq) *a = seq;
  if (*b > seq) *b = seq;
}

// Split-KV stage 1 for one query per request (decode: the query sits at
// position seq_i - 1 and sees every cached token).  partials is
// [N][Hq][S][d + 1]: the split's normalised output then its LSE.
template <typename E>
int split_partials(const E* q, const E* pool, const int32_t* block_table,
                   int max_blocks, const int32_t* seq_lens, int N, int Hq,
                   int Hkv, int d, int bs, int64_t nb, double scale, int S,
                   int64_t max_seq, double* partials, int threads) {
  if (Hkv <= 0 || Hq % Hkv != 0 || S <= 0 || bs <= 0) return -1;
  const int grp = Hq / Hkv;
  std::atomic<int> bad(0);
  parallel_for(static_cast<int64_t>(N) * Hkv, threads, [&](int64_t item) {
    const int i = static_cast<int>(item / Hkv);
    const int g = static_cast<int>(item % Hkv);
    const int64_t seq = seq_lens[i];
    std::vector<double> K, V, qv(d);
    if (!gather_standard(pool, block_table + static_cast<int64_t>(i) * max_blocks,
                         seq, g, Hkv, d, bs, nb, K, V)) {
      bad = 1;
      return;
    }
    for (int r = 0; r < grp; ++r) {
      const int h = g * grp + r;
      for (int e = 0; e < d; ++e) qv[e] = widen(q[(static_cast<int64_t>(i) * Hq + h) * d + e]);
      for (int s = 0; s < S; ++s) {
        int64_t a, b;
        split_range(seq, max_seq, S, bs, s, &a, &b);
        double* dst = partials + ((static_cast<int64_t>(i) * Hq + h) * S + s) * (d + 1);
        attend(qv.data(), K.data() + a * d, V.data() + a * d, b - a, d, d,
               scale, dst, dst + d);
      }
    }
  });
  return bad ? -1 : 0;
}

// MLA decode: one query per request, all H heads against the single latent
// KV head.  The key is the whole dk = kv_lora_rank + rope_dim row, the value
// its first kv_lora_rank entries.  pool is [nb][bs][dk].
template <typename E>
int mla_decode(const E* q, const E* pool, const int32_t* block_table,
               int max_blocks, const int32_t* seq_lens, int B, int H,
               int kv_lora_rank, int rope_dim, int bs, int64_t nb,
               double scale, const uint8_t* req_mask, double* out, double* lse,
               int threads) {
  const int dk = kv_lora_rank + rope_dim, dv = kv_lora_rank;
  if (bs <= 0 || dk <= 0) return -1;
  std::atomic<int> bad(0);
  parallel_for(B, threads, [&](int64_t b) {
    if (req_mask && !req_mask[b]) return;
    const int64_t seq = seq_lens[b];
    std::vector<double> K(static_cast<size_t>(seq) * dk), V(static_cast<size_t>(seq) * dv), qv(dk);
    const int32_t* row = block_table + b * max_blocks;
    for (int64_t p = 0; p < seq; ++p) {
      const int64_t blk = row[p / bs];
      if (blk < 0 || blk >= nb) {
        bad = 1;
        return;
      }
      const E* c = pool + (blk * bs + p % bs) * dk;
      for (int e = 0; e < dk; ++e) K[p * dk + e] = widen(c[e]);
      for (int e = 0; e < dv; ++e) V[p * dv + e] = widen(c[e]);
    }
    for (int h = 0; h < H; ++h) {
      for (int e = 0; e < dk; ++e) qv[e] = widen(q[(b * H + h) * dk + e]);
      attend(qv.data(), K.data(), V.data(), seq, dk, dv, scale,
             out + (b * H + h) * dv, lse + b * H + h);
    }
  });
  return bad ? -1 : 0;
}

// Nearest bf16 value of x (ties to even), in double: 8 significant bits.
double round_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e = std::ilogb(x);
  if (e < -126) e = -126;                        // bf16 subnormals: spacing 2^-133
  const double ulp = std::ldexp(1.0, e - 7);
  return std::nearbyint(x / ulp) * ulp;          // default rounding: to nearest even
}

// MLA prefill in the multi-head formulation ("Attention Backends", section
// "Latent attention is a different cache, not just a different kernel":
// prefill and decode use different formulations of the same mathematics;
// "AttentionBackend: attention backend abstraction layer": the MLA impl's
// entry points are forward_mqa for decode and forward_mha).  The cache holds [c | k_pe] per token (c: kv_lora_rank R,
// k_pe: rope_dim); the model's kv_b_proj weight w [H][dn + dv][R] expands c
// per head h into a key part k_nope = w[h][0:dn] c and a value
// v = w[h][dn:dn+dv] c.  Head h's key is [k_nope | k_pe] (dn + rope_dim),
// its value v; queries are [q_nope (dn) | q_pe (rope_dim)] per head.  With
// round_kv the expanded k_nope and v are rounded to bf16 (the dtype of the
// projection's output) before attention.  Causal alignment as in varlen.
template <typename E>
int mla_prefill(const E* q, const E* pool, const E* w, const int32_t* block_table,
                int max_blocks, const int32_t* qsl, const int32_t* seq_lens, int N, int H,
                int R, int dr, int dn, int dv, int bs, int64_t nb, double scale, int causal,
                int round_kv, const uint8_t* head_mask, const uint8_t* row_mask, double* out,
                double* lse, int threads) {
  if (bs <= 0 || R <= 0 || dn <= 0 || dv <= 0 || dr < 0) return -1;
  const int dk = dn + dr, wrow = dn + dv;
  std::atomic<int> bad(0);
  parallel_for(static_cast<int64_t>(N) * H, threads, [&](int64_t item) {
    const int i = static_cast<int>(item / H), h = static_cast<int>(item % H);
    if (head_mask && !head_mask[h]) return;
    const int64_t q0 = qsl[i], q1 = qsl[i + 1], seq = seq_lens[i], qlen = q1 - q0;
    if (qlen <= 0) return;
    if (qlen > seq) {
      bad = 1;
      return;
    }
    bool any = row_mask == nullptr;
    for (int64_t j = q0; j < q1 && !any; ++j) any = row_mask[j] != 0;
    if (!any) return;
    std::vector<double> C(static_cast<size_t>(R)), K(static_cast<size_t>(seq) * dk),
        V(static_cast<size_t>(seq) * dv), qv(dk);
    const int32_t* row = block_table + static_cast<int64_t>(i) * max_blocks;
    const E* wh = w + static_cast<int64_t>(h) * wrow * R;
    for (int64_t p = 0; p < seq; ++p) {
      const int64_t blk = row[p / bs];
      if (blk < 0 || blk >= nb) {
        bad = 1;
        return;
      }
      const E* c = pool + (blk * bs + p % bs) * (R + dr);
      for (int r = 0; r < R; ++r) C[r] = widen(c[r]);
      for (int e = 0; e < wrow; ++e) {
        double acc = 0.0;
        for (int r = 0; r < R; ++r) acc += widen(wh[static_cast<int64_t>(e) * R + r]) * C[r];
        if (round_kv) acc = round_bf16(acc);
        if (e < dn)
          K[p * dk + e] = acc;
        else
          V[p * dv + (e - dn)] = acc;
      }
      for (int e = 0; e < dr; ++e) K[p * dk + dn + e] = widen(c[R + e]);
    }
    const int64_t ctx = seq - qlen;
    for (int64_t j = q0; j < q1; ++j) {
      if (row_mask && !row_mask[j]) continue;
      const int64_t visible = causal ? ctx + (j - q0) + 1 : seq;
      for (int e = 0; e < dk; ++e) qv[e] = widen(q[(j * H + h) * dk + e]);
      attend(qv.data(), K.data(), V.data(), visible, dk, dv, scale, out + (j * H + h) * dv,
             lse + j * H + h);
    }
  });
  return bad ? -1 : 0;
}

}  // namespace

extern "C" {

// MLA prefill (multi-head formulation), bf16 inputs: q [T][H][dn + dr],
// pool [nb][bs][R + dr], w [H][dn + dv][R]; out [T][H][dv], lse [T][H] fp64.
// head_mask ([H]) and row_mask ([T]) are nullable selections.
int oracle_mla_prefill(const uint16_t* q, const uint16_t* pool, const uint16_t* w,
                       const int32_t* block_table, int max_blocks, const int32_t* qsl,
                       const int32_t* seq_lens, int N, int H, int R, int dr, int dn, int dv,
                       int bs, int64_t nb, double scale, int causal, int round_kv,
                       const uint8_t* head_mask, const uint8_t* row_mask, double* out,
                       double* lse, int threads) {
  return mla_prefill(q, pool, w, block_table, max_blocks, qsl, seq_lens, N, H, R, dr, dn, dv, bs,
                     nb, scale, causal, round_kv, head_mask, row_mask, out, lse, threads);
}

// Nearest bf16 values (ties to even) of n doubles, as doubles.
void oracle_round_bf16(const double* src, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = round_bf16(src[i]);
}

// Step 1 of the paged-kernel contract: for every token t with
// slot = slot_mapping[t] >= 0, copy key[t] / value[t] ([Hkv][d] each) into
// pool[slot / bs][0 or 1][slot % bs].  A bit copy of 16-bit elements.
// Returns -1 (and writes nothing more) on a slot outside the pool.
int oracle_reshape_and_cache(const uint16_t* key, const uint16_t* value,
                             uint16_t* pool, const int64_t* slot_mapping,
                             int64_t num_tokens, int num_kv_heads, int head_size,
                             int block_size, int64_t num_blocks) {
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_size;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size, off = slot % block_size;
    if (blk >= num_blocks) return -1;
    std::memcpy(pool + ((blk * 2 + 0) * block_size + off) * row, key + t * row,
                sizeof(uint16_t) * row);
    std::memcpy(pool + ((blk * 2 + 1) * block_size + off) * row, value + t * row,
                sizeof(uint16_t) * row);
  }
  return 0;
}

// The MLA cache write: a new token's cache entry is its compressed latent
// kv_c followed by its rotary key part k_pe, one kv_lora_rank + rope_dim
// vector per token, no K/V halves ("Triton and MLA": the cache holds the
// concatenation [kv_c (kv_lora_rank), k_pe (qk_rope_head_dim)]; its shape is
// (num_blocks, block_size, head_size)).  slot < 0 skips the token.
int oracle_mla_cache_write(const uint16_t* kv_c, const uint16_t* k_pe, uint16_t* pool,
                           const int64_t* slot_mapping, int64_t num_tokens, int kv_lora_rank,
                           int rope_dim, int block_size, int64_t num_blocks) {
  const int64_t width = static_cast<int64_t>(kv_lora_rank) + rope_dim;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size, off = slot % block_size;
    if (blk >= num_blocks) return -1;
    uint16_t* dst = pool + (blk * block_size + off) * width;
    std::memcpy(dst, kv_c + t * kv_lora_rank, sizeof(uint16_t) * kv_lora_rank);
    std::memcpy(dst + kv_lora_rank, k_pe + t * rope_dim, sizeof(uint16_t) * rope_dim);
  }
  return 0;
}

// Step 2 of the contract (varlen paged attention), bf16 inputs.
// q [T][Hq][d], pool [nb][2][bs][Hkv][d], out [T][Hq][d] fp64,
// lse [T][Hq] fp64 natural log.  row_mask (nullable, [T]) selects rows.
int oracle_paged_attention_bf16(const uint16_t* q, const uint16_t* pool,
                                const int32_t* block_table, int max_blocks,
                                const int32_t* query_start_loc,
                                const int32_t* seq_lens, int N, int Hq, int Hkv,
                                int d, int bs, int64_t nb, double scale,
                                int causal, int window, const uint8_t* row_mask,
                                double* out, double* lse, int threads) {
  return paged_attention(q, pool, block_table, max_blocks, query_start_loc,
                         seq_lens, N, Hq, Hkv, d, bs, nb, scale, causal, window,
                         row_mask, out, lse, threads);
}

// Same as above with fp64 q and pool (used by the worked-example pins).
int oracle_paged_attention_f64(const double* q, const double* pool,
                               const int32_t* block_table, int max_blocks,
                               const int32_t* query_start_loc,
                               const int32_t* seq_lens, int N, int Hq, int Hkv,
                               int d, int bs, int64_t nb, double scale,
                               int causal, int window, const uint8_t* row_mask,
                               double* out, double* lse, int threads) {
  return paged_attention(q, pool, block_table, max_blocks, query_start_loc,
                         seq_lens, N, Hq, Hkv, d, bs, nb, scale, causal, window,
                         row_mask, out, lse, threads);
}

// Split-KV stage 1 (decode, one query per request), bf16 / fp64 inputs.
// max_seq sizes the split chunk (see split_range).
int oracle_split_partials_bf16(const uint16_t* q, const uint16_t* pool,
                               const int32_t* block_table, int max_blocks,
                               const int32_t* seq_lens, int N, int Hq, int Hkv,
                               int d, int bs, int64_t nb, double scale,
                               int num_splits, int64_t max_seq, double* partials,
                               int threads) {
  return split_partials(q, pool, block_table, max_blocks, seq_lens, N, Hq, Hkv,
                        d, bs, nb, scale, num_splits, max_seq, partials, threads);
}
int oracle_split_partials_f64(const double* q, const double* pool,
                              const int32_t* block_table, int max_blocks,
                              const int32_t* seq_lens, int N, int Hq, int Hkv,
                              int d, int bs, int64_t nb, double scale,
                              int num_splits, int64_t max_seq, double* partials,
                              int threads) {
  return split_partials(q, pool, block_table, max_blocks, seq_lens, N, Hq, Hkv,
                        d, bs, nb, scale, num_splits, max_seq, partials, threads);
}

// Split-KV stage 2: merge S partials per (request, head) by their LSE.
// partials [N][H][S][dv + 1] -> out [N][H][dv], lse [N][H].
//   M = max_s lse_s, w_s = exp(lse_s - M), o = sum_s w_s o_s / sum_s w_s,
//   lse = M + ln(sum_s w_s).  All splits empty (M = -inf): o = 0, lse = -inf.
void oracle_lse_merge(const double* partials, int N, int H, int S, int dv,
                      double* out, double* lse) {
  for (int64_t nh = 0; nh < static_cast<int64_t>(N) * H; ++nh) {
    const double* base = partials + nh * S * (dv + 1);
    double m = kNegInf;
    for (int s = 0; s < S; ++s) {
      const double l = base[s * (dv + 1) + dv];
      if (l > m) m = l;
    }
    double* o = out + nh * dv;
    for (int e = 0; e < dv; ++e) o[e] = 0.0;
    if (m == kNegInf) {
      lse[nh] = kNegInf;
      continue;
    }
    double wsum = 0.0;
    for (int s = 0; s < S; ++s) {
      const double l = base[s * (dv + 1) + dv];
      if (l == kNegInf) continue;
      const double w = std::exp(l - m);
      wsum += w;
      for (int e = 0; e < dv; ++e) o[e] += w * base[s * (dv + 1) + e];
    }
    for (int e = 0; e < dv; ++e) o[e] /= wsum;
    lse[nh] = m + std::log(wsum);
  }
}

// MLA latent decode, bf16 / fp64 inputs.  q [B][H][dk], pool [nb][bs][dk],
// out [B][H][kv_lora_rank], lse [B][H].  req_mask (nullable, [B]).
int oracle_mla_decode_bf16(const uint16_t* q, const uint16_t* pool,
                           const int32_t* block_table, int max_blocks,
                           const int32_t* seq_lens, int B, int H,
                           int kv_lora_rank, int rope_dim, int bs, int64_t nb,
                           double scale, const uint8_t* req_mask, double* out,
                           double* lse, int threads) {
  return mla_decode(q, pool, block_table, max_blocks, seq_lens, B, H,
                    kv_lora_rank, rope_dim, bs, nb, scale, req_mask, out, lse,
                    threads);
}
int oracle_mla_decode_f64(const double* q, const double* pool,
                          const int32_t* block_table, int max_blocks,
                          const int32_t* seq_lens, int B, int H,
                          int kv_lora_rank, int rope_dim, int bs, int64_t nb,
                          double scale, const uint8_t* req_mask, double* out,
                          double* lse, int threads) {
  return mla_decode(q, pool, block_table, max_blocks, seq_lens, B, H,
                    kv_lora_rank, rope_dim, bs, nb, scale, req_mask, out, lse,
                    threads);
}

// Exact bf16 -> fp64 widening of n values (for callers that want the
// oracle's view of a bf16 array).
// ---------------------------------------------------------------- fp8 cache
// The pages ("Triton and MLA", data flow: decode_attention_fwd always gets
// the layer's k_scale / v_scale; "when the KV cache is BF16 the fp8 check is
// a no-op") give only the read side: an fp8 cache entry c stands for
// value(c) * scale.  The write side is read as its inverse: the code of a
// new key x is the e4m3 value nearest to x / k_scale (ties to even),
// computed in fp32 (the precision the quantising kernel works in), with
// magnitudes past the largest finite e4m3 value (448) saturating to it.
//
// e4m3 (OCP FP8, "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3
// mantissa bits; exponent 0 is subnormal (m * 2^-9); exponent 15 with
// mantissa 7 is NaN; there is no infinity.

double oracle_e4m3_value(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7)
    v = std::numeric_limits<double>::quiet_NaN();
  else if (e == 0)
    v = std::ldexp(static_cast<double>(m), -9);
  else
    v = std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

uint8_t oracle_e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 448.0) return sign | 0x7E;
  if (a < std::ldexp(1.0, -6)) {
    // Subnormal range: multiples of 2^-9 (m = 8 is the smallest normal).
    const double m = std::nearbyint(a / std::ldexp(1.0, -9));
    return sign | static_cast<uint8_t>(m);   // m <= 8 -> code 8 = 2^-6
  }
  int e2;
  std::frexp(a, &e2);                  // a = f * 2^e2, f in [0.5, 1)
  int e = e2 - 1;                      // a in [2^e, 2^(e+1))
  double m = std::nearbyint(a / std::ldexp(1.0, e - 3));   // 8 .. 16
  if (m >= 16.0) {
    m = 8.0;
    ++e;
  }
  const int field = e + 7;
  if (field > 15 || (field == 15 && m - 8.0 >= 7.0)) return sign | 0x7E;
  return sign | static_cast<uint8_t>((field << 3) | static_cast<int>(m - 8.0));
}

void oracle_e4m3_decode(const uint8_t* src, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = oracle_e4m3_value(src[i]);
}

void oracle_e4m3_encode_f32(const float* src, uint8_t* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = oracle_e4m3_encode(src[i]);
}

// Step 1 with an fp8 pool [nb][2][bs][Hkv][d] of e4m3 codes.
int oracle_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value, uint8_t* pool,
                                 const int64_t* slot_mapping, int64_t T, int Hkv, int d, int bs,
                                 int64_t nb, float k_scale, float v_scale) {
  const int64_t row = static_cast<int64_t>(Hkv) * d;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= nb * bs) return -1;
    const int64_t blk = slot / bs, off = slot % bs;
    uint8_t* kdst = pool + ((blk * 2 + 0) * bs + off) * row;
    uint8_t* vdst = pool + ((blk * 2 + 1) * bs + off) * row;
    for (int64_t e = 0; e < row; ++e) {
      const float kx = static_cast<float>(widen(key[t * row + e]));
      const float vx = static_cast<float>(widen(value[t * row + e]));
      kdst[e] = oracle_e4m3_encode(kx / k_scale);
      vdst[e] = oracle_e4m3_encode(vx / v_scale);
    }
  }
  return 0;
}

// The pool's values: K entries value(c) * k_scale, V entries value(c) *
// v_scale, in fp64 (exact: 4 significant bits times a float's 24).
void oracle_dequant_pool_fp8(const uint8_t* pool, int64_t nb, int bs, int Hkv, int d,
                             float k_scale, float v_scale, double* out) {
  const int64_t half = static_cast<int64_t>(bs) * Hkv * d;
  for (int64_t b = 0; b < nb; ++b)
    for (int kv = 0; kv < 2; ++kv) {
      const double sc = kv == 0 ? static_cast<double>(k_scale) : static_cast<double>(v_scale);
      const int64_t base = (b * 2 + kv) * half;
      for (int64_t e = 0; e < half; ++e) out[base + e] = oracle_e4m3_value(pool[base + e]) * sc;
    }
}

void oracle_bf16_to_f64(const uint16_t* src, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = widen(src[i]);
}

}  // extern "C"
