// Split-KV decode for callers that cannot allocate device memory.
//
// pa_decode_splitkv + pa_lse_merge need a caller-provided fp32 workspace.
// Some callers have no way to provide one: a host application that owns every
// device allocation and hands the library no allocator, or a code path that
// must never call cudaMalloc (which can synchronise the whole device).
// pa_decode_noalloc runs the same two kernels with the split partials in a
// fixed array in this file instead.
//
// The array is a file-scope __device__ variable: every device that loads the
// library holds its PA_NOALLOC_WORKSPACE_BYTES until the process exits.  Host
// code cannot use the array's name as a device address (on the host it names
// a stand-in object), so the first call on each device looks up the device
// address with cudaGetSymbolAddress while that device is current and caches
// it; make that first call before any stream capture begins.  Every call
// shares the one array: calls whose kernels may overlap on the GPU (different
// streams, no ordering between them) race on it.  Nothing needs clearing
// between calls -- stage 1 writes every partial it uses before the merge
// reads it.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"
#include "pa_common.cuh"
#include "pa_launch.h"


namespace {

constexpr size_t kNoallocFloats = PA_NOALLOC_WORKSPACE_BYTES / sizeof(float);

static __device__ __align__(256) float g_noalloc_workspace[kNoallocFloats];

// Device address of g_noalloc_workspace on the current device, looked up once
// per device.  nullptr if the lookup fails.
float* noalloc_workspace() {
  static std::mutex mu;
  static float* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cached[dev] != nullptr) return cached[dev];
  float* ptr = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_workspace) != cudaSuccess)
    return nullptr;
  if (dev < 64) cached[dev] = ptr;
  return ptr;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const void* q, const void* kv_cache,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       const pa_shape* shape, float scale, int num_splits,
                                       int max_seq_len, void* out, float* lse, void* stream) {
  if (shape == nullptr || shape->num_seqs < 0 || shape->num_q_heads <= 0 ||
      shape->num_kv_heads <= 0 || shape->head_size <= 0 || shape->block_size <= 0 ||
      shape->block_size % 16 != 0 || shape->num_blocks <= 0 || shape->max_blocks_per_seq <= 0 ||
      shape->num_q_heads % shape->num_kv_heads != 0 || shape->num_seqs > 65535 ||
      shape->num_kv_heads > 65535 || num_splits < 1 || num_splits > 16384 || max_seq_len < 0)
    return PA_ERR_INVALID;
  if (shape->head_size != 64 && shape->head_size != 128) return PA_ERR_UNSUPPORTED;
  if (shape->num_q_heads / shape->num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
  const size_t need = static_cast<size_t>(shape->num_seqs) * shape->num_q_heads * num_splits *
                      (static_cast<size_t>(shape->head_size) + 1);
  if (need > kNoallocFloats) return PA_ERR_INVALID;   // larger than the fixed array
  if (shape->num_seqs == 0) return PA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr || seq_lens == nullptr ||
      out == nullptr)
    return PA_ERR_INVALID;
  const uintptr_t qa = reinterpret_cast<uintptr_t>(q), ca = reinterpret_cast<uintptr_t>(kv_cache),
                  oa = reinterpret_cast<uintptr_t>(out), la = reinterpret_cast<uintptr_t>(lse);
  if (qa % 4 != 0 || ca % 16 != 0 || oa % 2 != 0 || la % 4 != 0) return PA_ERR_INVALID;
  float* ws = noalloc_workspace();
  if (ws == nullptr) return PA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = pa::launch_decode_splitkv(
      q, kv_cache, block_table, seq_lens, shape->num_seqs, shape->num_q_heads,
      shape->num_kv_heads, shape->head_size, shape->block_size, shape->num_blocks,
      shape->max_blocks_per_seq, scale, num_splits,
      static_cast<int>(pa::split_chunk(max_seq_len, num_splits, shape->block_size)), ws,
      pa::device_error_word(), st);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  e = pa::launch_lse_merge(ws, shape->num_seqs * shape->num_q_heads, num_splits,
                           shape->head_size, out, lse, st);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
