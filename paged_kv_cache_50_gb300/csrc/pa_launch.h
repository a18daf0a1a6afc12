// Host-side launchers of the library's kernels (one per .cu file), used by the
// C-ABI entry points.  Each returns the launch's cudaError_t.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (nullptr if the driver does not provide it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* cache,
                                     const int64_t* slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_size, int block_size,
                                     int num_blocks, int* err, cudaStream_t stream);

// Offsets of a split-KV stage-1 launch that serves part of a larger
// computation (the suffix pass of cascade attention): every request skips its
// first seq_off tokens, whose blocks are the first table_col0 columns of its
// row, and split s writes slot ws_slot0 + s of a workspace with ws_slots
// slots per (request, head).
struct DecodeExt {
  int table_col0;
  int seq_off;
  int ws_slots;
  int ws_slot0;
};

// Split-KV stage 1; `chunk` = tokens per split (split_chunk in pa_common.cuh).
// ext == nullptr: no offsets, S slots.
cudaError_t launch_decode_splitkv(const void* q, const void* cache, const int32_t* block_table,
                                  const int32_t* seq_lens, int N, int Hq, int Hkv, int d, int bs,
                                  int num_blocks, int max_blocks, float scale, int S, int chunk,
                                  float* ws, int* err, cudaStream_t stream,
                                  const DecodeExt* ext = nullptr);

// MLA cache write: [kv_c | k_pe] rows of a [nb, bs, kv_lora_rank + rope_dim] pool.
cudaError_t launch_mla_cache_write(const void* kv_c, const void* k_pe, void* cache,
                                   const int64_t* slot_mapping, int num_tokens, int kv_lora_rank,
                                   int rope_dim, int block_size, int num_blocks, int* err,
                                   cudaStream_t stream);

// MLA prefill, step 1: expand every context token's latent through kv_b_proj
// into K_ws [N][s_max][H][192] = [k_nope | k_pe] and V_ws [N][s_max][H][128]
// (bf16).  Fixed widths: kv_lora_rank 512, rope 64, nope 128, v 128.
cudaError_t launch_mla_expand(const void* pool, const void* w_kv_b, const int32_t* block_table,
                              const int32_t* seq_lens, int N, int H, int bs, int num_blocks,
                              int max_blocks, int max_seq_len, int s_max, void* k_ws, void* v_ws,
                              int* err, cudaStream_t stream);

// fp8 (e4m3) pool: quantising cache write and split-KV stage 1.
cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, void* cache,
                                         const int64_t* slot_mapping, int num_tokens,
                                         int num_kv_heads, int head_size, int block_size,
                                         int num_blocks, float k_scale, float v_scale, int* err,
                                         cudaStream_t stream);
cudaError_t launch_decode_splitkv_fp8(const void* q, const void* cache,
                                      const int32_t* block_table, const int32_t* seq_lens, int N,
                                      int Hq, int Hkv, int d, int bs, int num_blocks,
                                      int max_blocks, float scale, float k_scale, float v_scale,
                                      int S, int chunk, float* ws, int* err, cudaStream_t stream);

cudaError_t launch_lse_merge(const float* ws, int NH, int S, int dv, void* out, float* lse,
                             cudaStream_t stream);

// Varlen paged attention on tcgen05 tensor cores with TMA-gathered K/V.
struct VarlenLaunch {
  const void* q;
  const void* cache;
  const int32_t* block_table;
  const int32_t* qsl;
  const int32_t* seq_lens;
  int N, Hq, Hkv, d, bs, num_blocks, max_blocks, max_query_len;
  float scale;
  int causal;
  int window;              // > 0: sliding window of that many positions (causal)
  void* out;               // bf16 [T, Hq, d] (unused in partial mode)
  float* lse;              // [T, Hq], nullable (unused in partial mode)
  int* err;
  int table_col0 = 0;      // first table column of every request's row
  int seq_off = 0;         // tokens skipped at the front of every request
  int virt_total_q = 0;    // > 0: all rows [0, virt_total_q) as one request ...
  int virt_seq = 0;        // ... over virt_seq tokens of table row 0
  float* ws = nullptr;     // partial mode: fp32 [rows, Hq, ws_slots, d + 1]
  int ws_slots = 0;
  int ws_slot0 = 0;        // split s writes slot ws_slot0 + s
  int kv_splits = 1;
  int kv_chunk = 0;        // tokens per split, a multiple of 128
  // MLA prefill attention: keys [N * mla_s_max][Hkv][192] and values
  // [N * mla_s_max][Hkv][128] (the expanded workspaces) instead of the pool;
  // q is [T][Hkv][192], out [T][Hkv][128], one q head per kv head.
  const void* mla_k = nullptr;
  const void* mla_v = nullptr;
  int mla_s_max = 0;
};
cudaError_t launch_varlen_tc(const VarlenLaunch& L, cudaStream_t stream);

// MLA stage 1 on tcgen05 tensor cores + merge.
cudaError_t launch_mla_tc(const void* q, const void* cache, const int32_t* block_table,
                          const int32_t* seq_lens, int B, int H, int bs, int num_blocks,
                          int max_blocks, float scale, int S, int chunk, float* ws, void* out,
                          float* lse, int* err, cudaStream_t stream);

// Device address of the error word on the current device (nullptr on error).
int* device_error_word();

}  // namespace pa
