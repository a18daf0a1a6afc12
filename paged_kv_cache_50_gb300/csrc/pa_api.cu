// C-ABI entry points of libpa.so (declared in include/pa.h): host-side
// validation, split planning and kernel launches.  Nothing here allocates
// device memory or synchronises the host (except pa_get_device_error, which
// is a diagnostic).
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>

#include "pa.h"
#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

// The device error word (PA_DEVERR_* bits).  Kernels receive its address.
__device__ int g_device_error = 0;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace pa

namespace {

constexpr int kMaxSplits = 16384;   // the merge keeps S weights in shared memory
constexpr int kMaxGridYZ = 65535;

bool shape_ok(const pa_shape* s) {
  return s != nullptr && s->num_seqs >= 0 && s->num_q_heads > 0 && s->num_kv_heads > 0 &&
         s->head_size > 0 && s->block_size > 0 && s->num_blocks > 0 &&
         s->max_blocks_per_seq > 0 && s->num_q_heads % s->num_kv_heads == 0 &&
         s->block_size % 16 == 0 && s->num_seqs <= kMaxGridYZ && s->num_kv_heads <= kMaxGridYZ;
}

pa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// The kernels move cache rows and MLA queries in 16-byte vectors and q / out
// rows in 4-byte pairs.
bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Device address of the error word on the current device (looked up once per
// device; a host-side symbol is not a device address).
int* device_error_ptr() {
  static std::mutex mu;
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cached[dev] != nullptr) return cached[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, pa::g_device_error) != cudaSuccess) return nullptr;
  if (dev < 64) cached[dev] = static_cast<int*>(p);
  return static_cast<int*>(p);
}

}  // namespace

namespace pa {
// The error word's device address for kernels launched from other files.
int* device_error_word() { return device_error_ptr(); }
}  // namespace pa

namespace {

pa::VarlenLaunch varlen_launch(const void* q, const void* kv_cache, const int32_t* block_table,
                               const int32_t* qsl, const int32_t* seq_lens, int max_query_len,
                               const pa_shape* shape, float scale, int causal, int window,
                               void* out, float* lse) {
  pa::VarlenLaunch L{};
  L.q = q;
  L.cache = kv_cache;
  L.block_table = block_table;
  L.qsl = qsl;
  L.seq_lens = seq_lens;
  L.N = shape->num_seqs;
  L.Hq = shape->num_q_heads;
  L.Hkv = shape->num_kv_heads;
  L.d = shape->head_size;
  L.bs = shape->block_size;
  L.num_blocks = shape->num_blocks;
  L.max_blocks = shape->max_blocks_per_seq;
  L.max_query_len = max_query_len;
  L.scale = scale;
  L.causal = causal;
  L.window = window;
  L.out = out;
  L.lse = lse;
  L.err = device_error_ptr();
  return L;
}

}  // namespace

extern "C" {

pa_status pa_reshape_and_cache(const void* key, const void* value, void* kv_cache,
                               const int64_t* slot_mapping, int num_tokens,
                               const pa_shape* shape, void* stream) {
  if (shape == nullptr || num_tokens < 0) return PA_ERR_INVALID;
  if (shape->num_kv_heads <= 0 || shape->head_size <= 0 || shape->block_size <= 0 ||
      shape->block_size % 16 != 0 || shape->num_blocks <= 0)
    return PA_ERR_INVALID;
  if (shape->head_size % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (key == nullptr || value == nullptr || kv_cache == nullptr || slot_mapping == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_INVALID;
  return from_cuda(pa::launch_reshape_and_cache(key, value, kv_cache, slot_mapping, num_tokens,
                                                shape->num_kv_heads, shape->head_size,
                                                shape->block_size, shape->num_blocks,
                                                device_error_ptr(),
                                                static_cast<cudaStream_t>(stream)));
}

pa_status pa_mla_cache_write(const void* kv_c, const void* k_pe, void* kv_cache,
                             const int64_t* slot_mapping, int num_tokens, int kv_lora_rank,
                             int rope_dim, int block_size, int num_blocks, void* stream) {
  if (num_tokens < 0 || kv_lora_rank <= 0 || rope_dim < 0 || block_size <= 0 ||
      block_size % 16 != 0 || num_blocks <= 0)
    return PA_ERR_INVALID;
  if (kv_lora_rank % 8 != 0 || rope_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (kv_c == nullptr || (k_pe == nullptr && rope_dim > 0) || kv_cache == nullptr ||
      slot_mapping == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(kv_c, 16) || !aligned(k_pe, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_INVALID;
  return from_cuda(pa::launch_mla_cache_write(kv_c, k_pe, kv_cache, slot_mapping, num_tokens,
                                              kv_lora_rank, rope_dim, block_size, num_blocks,
                                              device_error_ptr(),
                                              static_cast<cudaStream_t>(stream)));
}

size_t pa_mla_prefill_workspace_bytes(int num_seqs, int max_seq_len, int num_heads) {
  if (num_seqs < 0 || max_seq_len < 0 || num_heads <= 0) return 0;
  return static_cast<size_t>(num_seqs) * max_seq_len * num_heads * (192 + 128) * 2;
}

static bool mla_prefill_shape_ok(int num_seqs, int num_heads, int block_size, int num_blocks,
                                 int max_blocks_per_seq, int max_seq_len) {
  return num_seqs >= 0 && num_seqs <= kMaxGridYZ && num_heads > 0 && num_heads <= kMaxGridYZ &&
         block_size > 0 && block_size % 16 == 0 && num_blocks > 0 && max_blocks_per_seq > 0 &&
         max_seq_len >= 0;
}

pa_status pa_mla_expand_kv(const void* kv_cache, const void* w_kv_b, const int32_t* block_table,
                           const int32_t* seq_lens, int num_seqs, int num_heads, int block_size,
                           int num_blocks, int max_blocks_per_seq, int max_seq_len, void* k_ws,
                           void* v_ws, void* stream) {
  if (!mla_prefill_shape_ok(num_seqs, num_heads, block_size, num_blocks, max_blocks_per_seq,
                            max_seq_len))
    return PA_ERR_INVALID;
  if (num_seqs == 0 || max_seq_len == 0) return PA_OK;
  if (kv_cache == nullptr || w_kv_b == nullptr || block_table == nullptr ||
      seq_lens == nullptr || k_ws == nullptr || v_ws == nullptr)
    return PA_ERR_INVALID;
  // The expansion writes its rows with 32-byte stores.
  if (!aligned(kv_cache, 16) || !aligned(w_kv_b, 16) || !aligned(k_ws, 32) || !aligned(v_ws, 32))
    return PA_ERR_INVALID;
  return from_cuda(pa::launch_mla_expand(kv_cache, w_kv_b, block_table, seq_lens, num_seqs,
                                         num_heads, block_size, num_blocks, max_blocks_per_seq,
                                         max_seq_len, max_seq_len, k_ws, v_ws,
                                         device_error_ptr(), static_cast<cudaStream_t>(stream)));
}

pa_status pa_mla_prefill(const void* q, const void* kv_cache, const void* w_kv_b,
                         const int32_t* block_table, const int32_t* query_start_loc,
                         const int32_t* seq_lens, int total_q, int max_query_len, int num_seqs,
                         int num_heads, int block_size, int num_blocks, int max_blocks_per_seq,
                         int max_seq_len, float scale, int causal, void* workspace, void* out,
                         float* lse, void* stream) {
  if (!mla_prefill_shape_ok(num_seqs, num_heads, block_size, num_blocks, max_blocks_per_seq,
                            max_seq_len) ||
      total_q < 0 || max_query_len < 0)
    return PA_ERR_INVALID;
  if (total_q == 0 || num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || w_kv_b == nullptr || block_table == nullptr ||
      query_start_loc == nullptr || seq_lens == nullptr || workspace == nullptr || out == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(w_kv_b, 16) ||
      !aligned(workspace, 32) || !aligned(out, 16) || !aligned(lse, 4))
    return PA_ERR_INVALID;
  const long long rows = static_cast<long long>(num_seqs) * max_seq_len;
  if (rows * num_heads > INT_MAX) return PA_ERR_INVALID;   // 3-D map row coordinate
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* k_ws = static_cast<uint8_t*>(workspace);
  uint8_t* v_ws = k_ws + rows * num_heads * 192 * 2;
  if (pa::launch_mla_expand(kv_cache, w_kv_b, block_table, seq_lens, num_seqs, num_heads,
                            block_size, num_blocks, max_blocks_per_seq, max_seq_len, max_seq_len,
                            k_ws, v_ws, device_error_ptr(), st) != cudaSuccess)
    return PA_ERR_CUDA;
  pa::VarlenLaunch L{};
  L.q = q;
  L.cache = kv_cache;
  L.block_table = block_table;
  L.qsl = query_start_loc;
  L.seq_lens = seq_lens;
  L.N = num_seqs;
  L.Hq = num_heads;
  L.Hkv = num_heads;
  L.d = 192;
  L.bs = block_size;
  L.num_blocks = num_blocks;
  L.max_blocks = max_blocks_per_seq;
  L.max_query_len = max_query_len;
  L.scale = scale;
  L.causal = causal ? 1 : 0;
  L.window = 0;
  L.out = out;
  L.lse = lse;
  L.err = device_error_ptr();
  L.mla_k = k_ws;
  L.mla_v = v_ws;
  L.mla_s_max = max_seq_len;
  return from_cuda(pa::launch_varlen_tc(L, st));
}

pa_status pa_varlen_fwd(const void* q, const void* kv_cache, const int32_t* block_table,
                        const int32_t* query_start_loc, const int32_t* seq_lens, int total_q,
                        int max_query_len, const pa_shape* shape, float scale, int causal,
                        void* out, float* lse, void* stream) {
  if (!shape_ok(shape) || total_q < 0 || max_query_len < 0) return PA_ERR_INVALID;
  if (shape->head_size != 64 && shape->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (total_q == 0 || shape->num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr ||
      query_start_loc == nullptr || seq_lens == nullptr || out == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return PA_ERR_INVALID;
  return from_cuda(pa::launch_varlen_tc(
      varlen_launch(q, kv_cache, block_table, query_start_loc, seq_lens, max_query_len, shape,
                    scale, causal ? 1 : 0, 0, out, lse),
      static_cast<cudaStream_t>(stream)));
}

pa_status pa_varlen_fwd_window(const void* q, const void* kv_cache, const int32_t* block_table,
                               const int32_t* query_start_loc, const int32_t* seq_lens,
                               int total_q, int max_query_len, const pa_shape* shape, float scale,
                               int sliding_window, void* out, float* lse, void* stream) {
  if (!shape_ok(shape) || total_q < 0 || max_query_len < 0 || sliding_window < 1)
    return PA_ERR_INVALID;
  if (shape->head_size != 64 && shape->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (total_q == 0 || shape->num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr ||
      query_start_loc == nullptr || seq_lens == nullptr || out == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return PA_ERR_INVALID;
  return from_cuda(pa::launch_varlen_tc(
      varlen_launch(q, kv_cache, block_table, query_start_loc, seq_lens, max_query_len, shape,
                    scale, 1, sliding_window, out, lse),
      static_cast<cudaStream_t>(stream)));
}

int pa_cascade_prefix_splits(int total_q, int num_q_heads, int num_kv_heads,
                             int prefix_tokens, int sm_count) {
  if (total_q <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || prefix_tokens <= 0) return 1;
  if (sm_count <= 0) sm_count = pa_device_sm_count();
  if (sm_count <= 0) sm_count = 1;
  // One CTA per (256 packed rows, kv head, split) and one CTA per SM: split
  // the prefix until every SM has a unit, at most one split per 128 tokens.
  const long long rows = static_cast<long long>(total_q) * (num_q_heads / num_kv_heads);
  const long long units = ((rows + 255) / 256) * num_kv_heads;
  long long s = (sm_count + units - 1) / units;
  const long long by_len = (static_cast<long long>(prefix_tokens) + 127) / 128;
  if (s > by_len) s = by_len;
  if (s > kMaxSplits - 1) s = kMaxSplits - 1;
  return s < 1 ? 1 : static_cast<int>(s);
}

pa_status pa_cascade_fwd(const void* q, const void* kv_cache, const int32_t* block_table,
                         const int32_t* query_start_loc, const int32_t* seq_lens, int total_q,
                         int max_query_len, int max_seq_len, int num_common_prefix_blocks,
                         int num_prefix_splits, int num_suffix_splits, const pa_shape* shape,
                         float scale, int causal, float* workspace, void* out, float* lse,
                         void* stream) {
  if (!shape_ok(shape) || total_q < 0 || max_query_len < 0 || max_seq_len < 0 ||
      num_common_prefix_blocks < 0 || num_common_prefix_blocks > shape->max_blocks_per_seq ||
      num_prefix_splits < 1 || num_suffix_splits < 1 ||
      num_prefix_splits + num_suffix_splits > kMaxSplits)
    return PA_ERR_INVALID;
  if (shape->head_size != 64 && shape->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (shape->num_q_heads / shape->num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
  if (total_q == 0 || shape->num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr ||
      query_start_loc == nullptr || seq_lens == nullptr || out == nullptr || workspace == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(workspace, 4))
    return PA_ERR_INVALID;
  const long long prefix_tokens =
      static_cast<long long>(num_common_prefix_blocks) * shape->block_size;
  const long long nh = static_cast<long long>(total_q) * shape->num_q_heads;
  if (prefix_tokens > INT_MAX || nh > INT_MAX) return PA_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (prefix_tokens == 0)   // nothing shared: plain varlen attention
    return from_cuda(pa::launch_varlen_tc(
        varlen_launch(q, kv_cache, block_table, query_start_loc, seq_lens, max_query_len, shape,
                      scale, causal ? 1 : 0, 0, out, lse),
        st));
  const int slots = num_prefix_splits + num_suffix_splits;
  {
    // Pass 1: every query row of the batch against the shared prefix (read
    // through row 0 of the table), no mask, cut into num_prefix_splits
    // pieces: slots [0, num_prefix_splits).
    pa::VarlenLaunch L = varlen_launch(q, kv_cache, block_table, query_start_loc, seq_lens,
                                       max_query_len, shape, scale, 0, 0, out, lse);
    L.virt_total_q = total_q;
    L.virt_seq = static_cast<int>(prefix_tokens);
    L.ws = workspace;
    L.ws_slots = slots;
    L.ws_slot0 = 0;
    L.kv_splits = num_prefix_splits;
    const long long per = (prefix_tokens + num_prefix_splits - 1) / num_prefix_splits;
    L.kv_chunk = static_cast<int>((per + 127) / 128 * 128);
    if (pa::launch_varlen_tc(L, st) != cudaSuccess) return PA_ERR_CUDA;
  }
  // Pass 2: each request against its own blocks after the prefix (positions
  // shift alike for keys and queries, so the call's mask is kept), cut into
  // num_suffix_splits pieces: slots [num_prefix_splits, slots).  A batch of
  // one query per request takes the split-KV decode kernel.
  const int suffix_max = static_cast<int>(std::max(0LL, max_seq_len - prefix_tokens));
  if (max_query_len == 1 && total_q == shape->num_seqs) {
    const pa::DecodeExt ext{num_common_prefix_blocks, static_cast<int>(prefix_tokens), slots,
                            num_prefix_splits};
    if (pa::launch_decode_splitkv(
            q, kv_cache, block_table, seq_lens, shape->num_seqs, shape->num_q_heads,
            shape->num_kv_heads, shape->head_size, shape->block_size, shape->num_blocks,
            shape->max_blocks_per_seq, scale, num_suffix_splits,
            static_cast<int>(pa::split_chunk(suffix_max, num_suffix_splits, shape->block_size)),
            workspace, device_error_ptr(), st, &ext) != cudaSuccess)
      return PA_ERR_CUDA;
  } else {
    pa::VarlenLaunch L2 = varlen_launch(q, kv_cache, block_table, query_start_loc, seq_lens,
                                        max_query_len, shape, scale, causal ? 1 : 0, 0, out, lse);
    L2.table_col0 = num_common_prefix_blocks;
    L2.seq_off = static_cast<int>(prefix_tokens);
    L2.ws = workspace;
    L2.ws_slots = slots;
    L2.ws_slot0 = num_prefix_splits;
    L2.kv_splits = num_suffix_splits;
    const long long per = (static_cast<long long>(suffix_max) + num_suffix_splits - 1) /
                          num_suffix_splits;
    L2.kv_chunk = static_cast<int>(std::max(128LL, (per + 127) / 128 * 128));
    if (pa::launch_varlen_tc(L2, st) != cudaSuccess) return PA_ERR_CUDA;
  }
  // Merge the partials by their LSE (the split-KV stage 2).
  return from_cuda(pa::launch_lse_merge(workspace, static_cast<int>(nh), slots,
                                        shape->head_size, out, lse, st));
}

int pa_device_sm_count(void) {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cached[dev] = sms;
  return sms;
}

int pa_num_kv_splits(int max_seq_len, int sm_count) {
  if (sm_count <= 0) sm_count = pa_device_sm_count();
  if (sm_count <= 0) sm_count = 1;
  const long long by_len = (static_cast<long long>(max_seq_len > 0 ? max_seq_len : 0) + 511) / 512;
  long long s = by_len < 2LL * sm_count ? by_len : 2LL * sm_count;
  if (s < 1) s = 1;
  if (s > kMaxSplits) s = kMaxSplits;
  return static_cast<int>(s);
}

int pa_decode_num_kv_splits(int num_seqs, int num_kv_heads, int max_seq_len, int sm_count) {
  if (num_seqs <= 0 || num_kv_heads <= 0) return 1;
  if (sm_count <= 0) sm_count = pa_device_sm_count();
  if (sm_count <= 0) sm_count = 1;
  const long long units = static_cast<long long>(num_seqs) * num_kv_heads;
  long long s = (12LL * sm_count + units - 1) / units;
  const int page = pa_num_kv_splits(max_seq_len, sm_count);
  if (s > page) s = page;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

int pa_mla_num_kv_splits(int batch, int num_heads, int max_seq_len, int sm_count) {
  if (batch <= 0 || num_heads <= 0) return 1;
  if (sm_count <= 0) sm_count = pa_device_sm_count();
  if (sm_count <= 0) sm_count = 1;
  const long long units = static_cast<long long>(batch) * ((num_heads + 127) / 128);
  const long long pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
  long long s = (pairs + units - 1) / units;
  const long long by_len = (static_cast<long long>(max_seq_len > 0 ? max_seq_len : 0) + 511) / 512;
  if (s > by_len) s = by_len;
  if (s < 1) s = 1;
  if (s > kMaxSplits) s = kMaxSplits;
  return static_cast<int>(s);
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_splits, int dv) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_splits <= 0 || dv <= 0) return 0;
  return static_cast<size_t>(num_seqs) * num_q_heads * num_splits * (static_cast<size_t>(dv) + 1) *
         sizeof(float);
}

pa_status pa_decode_splitkv(const void* q, const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, const pa_shape* shape, float scale,
                            int num_splits, int max_seq_len, float* workspace, void* stream) {
  if (!shape_ok(shape) || num_splits < 1 || num_splits > kMaxSplits || max_seq_len < 0)
    return PA_ERR_INVALID;
  if (shape->head_size != 64 && shape->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (shape->num_q_heads / shape->num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
  if (shape->num_seqs == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr || seq_lens == nullptr ||
      workspace == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(q, 4) || !aligned(kv_cache, 16) || !aligned(workspace, 4)) return PA_ERR_INVALID;
  return from_cuda(pa::launch_decode_splitkv(
      q, kv_cache, block_table, seq_lens, shape->num_seqs, shape->num_q_heads,
      shape->num_kv_heads, shape->head_size, shape->block_size, shape->num_blocks,
      shape->max_blocks_per_seq, scale, num_splits,
      static_cast<int>(pa::split_chunk(max_seq_len, num_splits, shape->block_size)), workspace,
      device_error_ptr(),
      static_cast<cudaStream_t>(stream)));
}

static bool scale_ok(float x) { return x > 0.f && x <= 3.4028234663852886e38f; }

pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* kv_cache,
                                   const int64_t* slot_mapping, int num_tokens,
                                   const pa_shape* shape, float k_scale, float v_scale,
                                   void* stream) {
  if (shape == nullptr || num_tokens < 0) return PA_ERR_INVALID;
  if (shape->num_kv_heads <= 0 || shape->head_size <= 0 || shape->block_size <= 0 ||
      shape->block_size % 16 != 0 || shape->num_blocks <= 0)
    return PA_ERR_INVALID;
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_ERR_INVALID;
  if (shape->head_size % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (key == nullptr || value == nullptr || kv_cache == nullptr || slot_mapping == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_INVALID;
  return from_cuda(pa::launch_reshape_and_cache_fp8(
      key, value, kv_cache, slot_mapping, num_tokens, shape->num_kv_heads, shape->head_size,
      shape->block_size, shape->num_blocks, k_scale, v_scale, device_error_ptr(),
      static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_splitkv_fp8(const void* q, const void* kv_cache, const int32_t* block_table,
                                const int32_t* seq_lens, const pa_shape* shape, float scale,
                                float k_scale, float v_scale, int num_splits, int max_seq_len,
                                float* workspace, void* stream) {
  if (!shape_ok(shape) || num_splits < 1 || num_splits > kMaxSplits || max_seq_len < 0)
    return PA_ERR_INVALID;
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_ERR_INVALID;
  if (shape->head_size != 64 && shape->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (shape->num_q_heads / shape->num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
  if (shape->num_seqs == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr || seq_lens == nullptr ||
      workspace == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(q, 4) || !aligned(kv_cache, 16) || !aligned(workspace, 4)) return PA_ERR_INVALID;
  return from_cuda(pa::launch_decode_splitkv_fp8(
      q, kv_cache, block_table, seq_lens, shape->num_seqs, shape->num_q_heads,
      shape->num_kv_heads, shape->head_size, shape->block_size, shape->num_blocks,
      shape->max_blocks_per_seq, scale, k_scale, v_scale, num_splits,
      static_cast<int>(pa::split_chunk(max_seq_len, num_splits, shape->block_size)), workspace,
      device_error_ptr(), static_cast<cudaStream_t>(stream)));
}

pa_status pa_lse_merge(const float* workspace, int num_seqs, int num_q_heads, int num_splits,
                       int dv, void* out, float* lse, void* stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_splits < 1 || num_splits > kMaxSplits || dv <= 0)
    return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (workspace == nullptr || out == nullptr) return PA_ERR_INVALID;
  if (!aligned(workspace, 4) || !aligned(out, 2) || !aligned(lse, 4)) return PA_ERR_INVALID;
  const long long nh = static_cast<long long>(num_seqs) * num_q_heads;
  if (nh > INT_MAX) return PA_ERR_INVALID;
  return from_cuda(pa::launch_lse_merge(workspace, static_cast<int>(nh), num_splits, dv, out, lse,
                                        static_cast<cudaStream_t>(stream)));
}

pa_status pa_mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                        const int32_t* seq_lens, int batch, int num_heads, int kv_lora_rank,
                        int rope_dim, int block_size, int num_blocks, int max_blocks_per_seq,
                        int max_seq_len, float scale, int num_splits, float* workspace, void* out,
                        float* lse,
                        void* stream) {
  if (batch < 0 || num_heads <= 0 || kv_lora_rank <= 0 || rope_dim < 0 || block_size <= 0 ||
      block_size % 16 != 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || num_splits < 1 ||
      num_splits > kMaxSplits || batch > kMaxGridYZ || num_splits > kMaxGridYZ || max_seq_len < 0)
    return PA_ERR_INVALID;
  if (kv_lora_rank != 512 || rope_dim != 64 || num_heads % 64 != 0 || block_size % 32 != 0)
    return PA_ERR_UNSUPPORTED;
  if (batch == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr || seq_lens == nullptr ||
      workspace == nullptr || out == nullptr)
    return PA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(workspace, 4) || !aligned(out, 2) ||
      !aligned(lse, 4))
    return PA_ERR_INVALID;
  return from_cuda(pa::launch_mla_tc(q, kv_cache, block_table, seq_lens, batch, num_heads,
                                         block_size, num_blocks, max_blocks_per_seq, scale,
                                         num_splits,
                                         static_cast<int>(pa::split_chunk(max_seq_len, num_splits,
                                                                          block_size)),
                                         workspace, out, lse, device_error_ptr(),
                                         static_cast<cudaStream_t>(stream)));
}

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: configuration not built";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA launch or query failed";
  }
  return "unknown pa_status";
}

pa_status pa_get_device_error(int* code, void* stream) {
  if (code == nullptr) return PA_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, pa::g_device_error, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(pa::g_device_error, &zero, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
  *code = v;
  return PA_OK;
}

}  // extern "C"
