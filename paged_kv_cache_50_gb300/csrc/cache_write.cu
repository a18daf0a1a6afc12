// Cache write: step 1 of the paged-kernel contract ("Attention Backends",
// section "What 'paged attention' requires of a kernel"): scatter the step's
// new keys and values into the block pool at slot_mapping.
//
// Pool layout [num_blocks, 2, block_size, Hkv, d]: for a fixed (block, K|V,
// offset) the [Hkv, d] slab is contiguous, so one token is two contiguous
// copies of Hkv*d*2 bytes.  One CTA per token, one 16-byte vector per thread
// per step; every byte is read once and written once (HBM-bound).
#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                         uint4* __restrict__ cache, const int64_t* __restrict__ slot_mapping,
                         int row_vec, int block_size, int64_t num_slots, int* err) {
  // The attention kernel that follows may start setting up now (it waits for
  // this kernel's completion before reading anything).
  pdl_trigger();
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) record_error(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / block_size, off = slot % block_size;
  uint4* kdst = cache + ((blk * 2 + 0) * block_size + off) * row_vec;
  uint4* vdst = cache + ((blk * 2 + 1) * block_size + off) * row_vec;
  const uint4* ksrc = key + static_cast<int64_t>(t) * row_vec;
  const uint4* vsrc = value + static_cast<int64_t>(t) * row_vec;
  for (int c = threadIdx.x; c < row_vec; c += blockDim.x) {
    const uint4 kv = __ldcs(ksrc + c);
    const uint4 vv = __ldcs(vsrc + c);
    kdst[c] = kv;
    vdst[c] = vv;
  }
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* cache,
                                     const int64_t* slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_size, int block_size,
                                     int num_blocks, int* err, cudaStream_t stream) {
  const int row_vec = num_kv_heads * head_size / 8;  // 16-byte vectors per row
  int threads = ((row_vec + 31) / 32) * 32;
  if (threads > 256) threads = 256;
  reshape_and_cache_kernel<<<num_tokens, threads, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value),
      static_cast<uint4*>(cache), slot_mapping, row_vec, block_size,
      static_cast<int64_t>(num_blocks) * block_size, err);
  return cudaGetLastError();
}

}  // namespace pa
