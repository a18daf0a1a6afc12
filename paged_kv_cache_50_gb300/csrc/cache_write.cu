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
  // Launched with launch_pdl: wait for the previous kernel in the stream
  // (which may still read the pool or produce these inputs) to complete.
  pdl_wait();
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
  return launch_pdl(reshape_and_cache_kernel, dim3(num_tokens), dim3(threads), 0, stream,
                    static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                    static_cast<uint4*>(cache), slot_mapping, row_vec, block_size,
                    static_cast<int64_t>(num_blocks) * block_size, err);
}

// The same step with an fp8 pool of e4m3 codes, [num_blocks, 2, block_size,
// Hkv, d] bytes ("Triton and MLA", data flow: the decode kernel always
// receives the layer's k_scale / v_scale, an fp8 entry standing for its
// e4m3 value times the scale).  The code of a new element x is the e4m3 value
// nearest to x / scale, the quotient taken in fp32 with IEEE rounding and the
// conversion rounding to nearest-even and saturating at +-448.  One thread
// turns 16 bf16 elements (two 16-byte loads) into one 16-byte store.
__device__ __forceinline__ uint32_t quant4(uint2 v, float scale) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint32_t r = 0;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    const float2 qv = make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3);
    r |= static_cast<uint32_t>(c) << (16 * k);
  }
  return r;
}

__device__ __forceinline__ uint4 quant16(uint4 a, uint4 b, float scale) {
  uint4 r;
  r.x = quant4(make_uint2(a.x, a.y), scale);
  r.y = quant4(make_uint2(a.z, a.w), scale);
  r.z = quant4(make_uint2(b.x, b.y), scale);
  r.w = quant4(make_uint2(b.z, b.w), scale);
  return r;
}

__global__ void __launch_bounds__(256)
reshape_and_cache_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             uint4* __restrict__ cache, const int64_t* __restrict__ slot_mapping,
                             int row_vec, int block_size, int64_t num_slots, float k_scale,
                             float v_scale, int* err) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0) record_error(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / block_size, off = slot % block_size;
  // row_vec = 16-byte vectors of codes per row; the bf16 source row has twice as many.
  uint4* kdst = cache + ((blk * 2 + 0) * block_size + off) * row_vec;
  uint4* vdst = cache + ((blk * 2 + 1) * block_size + off) * row_vec;
  const uint4* ksrc = key + static_cast<int64_t>(t) * row_vec * 2;
  const uint4* vsrc = value + static_cast<int64_t>(t) * row_vec * 2;
  for (int c = threadIdx.x; c < row_vec; c += blockDim.x) {
    const uint4 k0 = __ldcs(ksrc + 2 * c), k1 = __ldcs(ksrc + 2 * c + 1);
    const uint4 v0 = __ldcs(vsrc + 2 * c), v1 = __ldcs(vsrc + 2 * c + 1);
    kdst[c] = quant16(k0, k1, k_scale);
    vdst[c] = quant16(v0, v1, v_scale);
  }
}

cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, void* cache,
                                         const int64_t* slot_mapping, int num_tokens,
                                         int num_kv_heads, int head_size, int block_size,
                                         int num_blocks, float k_scale, float v_scale, int* err,
                                         cudaStream_t stream) {
  const int row_vec = num_kv_heads * head_size / 16;  // 16-byte vectors of codes per row
  int threads = ((row_vec + 31) / 32) * 32;
  if (threads > 256) threads = 256;
  return launch_pdl(reshape_and_cache_fp8_kernel, dim3(num_tokens), dim3(threads), 0, stream,
                    static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                    static_cast<uint4*>(cache), slot_mapping, row_vec, block_size,
                    static_cast<int64_t>(num_blocks) * block_size, k_scale, v_scale, err);
}

// The MLA cache write ("Triton and MLA": the cache holds one vector per token,
// [kv_c (kv_lora_rank) | k_pe (rope_dim)], in a [num_blocks, block_size,
// kv_lora_rank + rope_dim] pool).  One warp per token copies the two parts in
// 16-byte vectors into the row at slot_mapping.
__global__ void __launch_bounds__(128)
mla_cache_write_kernel(const uint4* __restrict__ kv_c, const uint4* __restrict__ k_pe,
                       uint4* __restrict__ cache, const int64_t* __restrict__ slot_mapping,
                       int num_tokens, int c_vec, int pe_vec, int64_t num_slots, int* err) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= num_tokens) return;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) record_error(err, PA_DEVERR_SLOT);
    return;
  }
  const int row_vec = c_vec + pe_vec;
  uint4* dst = cache + slot * row_vec;   // slot = block * block_size + offset
  const uint4* src_c = kv_c + static_cast<int64_t>(t) * c_vec;
  const uint4* src_pe = k_pe + static_cast<int64_t>(t) * pe_vec;
  for (int c = lane; c < row_vec; c += 32)
    dst[c] = c < c_vec ? __ldcs(src_c + c) : __ldcs(src_pe + (c - c_vec));
}

cudaError_t launch_mla_cache_write(const void* kv_c, const void* k_pe, void* cache,
                                   const int64_t* slot_mapping, int num_tokens, int kv_lora_rank,
                                   int rope_dim, int block_size, int num_blocks, int* err,
                                   cudaStream_t stream) {
  const int blocks = (num_tokens + 3) / 4;
  return launch_pdl(mla_cache_write_kernel, dim3(blocks), dim3(128), 0, stream,
                    static_cast<const uint4*>(kv_c), static_cast<const uint4*>(k_pe),
                    static_cast<uint4*>(cache), slot_mapping, num_tokens, kv_lora_rank / 8,
                    rope_dim / 8, static_cast<int64_t>(num_blocks) * block_size, err);
}

}  // namespace pa
