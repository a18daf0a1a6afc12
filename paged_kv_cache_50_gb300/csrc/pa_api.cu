// C-ABI entry points of libpa.so (declared in include/pa.h): host-side
// validation, split planning and kernel launches.  Nothing here allocates
// device memory or synchronises the host (except pa_get_device_error, which
// is a diagnostic).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "pa.h"
#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

// The device error word (PA_DEVERR_* bits).  Kernels receive its address.
__device__ int g_device_error = 0;

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
      q, kv_cache, block_table, query_start_loc, seq_lens, shape->num_seqs, shape->num_q_heads,
      shape->num_kv_heads, shape->head_size, shape->block_size, shape->num_blocks,
      shape->max_blocks_per_seq, max_query_len, scale, causal ? 1 : 0, out, lse,
      device_error_ptr(), static_cast<cudaStream_t>(stream)));
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
