// Shared device helpers for the paged-attention kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Device error word: PA_DEVERR_* bits, set by kernels that meet an index they
// refuse to dereference.  Every kernel gets its address as a parameter (the
// word lives in pa_api.cu and is read and cleared by pa_get_device_error).
__device__ __forceinline__ void record_error(int* err, int bit) {
  if (err != nullptr) atomicOr(err, bit);
}

// Block id of logical block `idx` of a request's table row; a column past the
// row (a seq_len longer than the table allows) reads as an invalid id (-1).
// log2(bs) if the block size is a power of two, else -1: the decode kernels
// then split a token index into (block, offset) with a shift and a mask
// instead of an integer division per 16-token sub-block.
inline int block_size_log2(int bs) {
  return (bs > 0 && (bs & (bs - 1)) == 0) ? __builtin_ctz(static_cast<unsigned>(bs)) : -1;
}
__device__ __forceinline__ int div_bs(int x, int bs, int bs_log2) {
  return bs_log2 >= 0 ? (x >> bs_log2) : x / bs;
}
__device__ __forceinline__ int mod_bs(int x, int bs, int bs_log2) {
  return bs_log2 >= 0 ? (x & (bs - 1)) : x % bs;
}

__device__ __forceinline__ int block_at(const int32_t* row, int idx, int max_blocks) {
  return idx < max_blocks ? __ldg(row + idx) : -1;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy; src_bytes == 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with f16 operands (used where K/V arrive as e4m3 codes, which
// f16 holds exactly).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// Per-device "done" flags for one-time host set-up.
// Programmatic dependent launch.  A kernel launched with launch_pdl may
// start while the previous kernel in its stream is still running (once every
// CTA of that kernel has called pdl_trigger or exited); it must call
// pdl_wait, which returns when that kernel has completed and its writes are
// visible, before it reads any input from global memory.  Both are no-ops
// for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct DeviceFlags {
  bool done[64] = {};
};

// Raises `kern`'s dynamic shared memory limit to `bytes` once per device.
template <typename Kernel>
inline cudaError_t set_smem_once(Kernel kern, int bytes, DeviceFlags& flags) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && flags.done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) flags.done[dev] = true;
  return e;
}

// Tokens per split: the sequence axis of every request is cut at multiples
// of chunk = bs * ceil(ceil(max_seq_len / S) / bs) (the last split of a
// request runs to its end).
inline long long split_chunk(int max_seq_len, int S, int bs) {
  const long long m = max_seq_len > 0 ? max_seq_len : 1;
  const long long per = (m + S - 1) / S;
  return ((per + bs - 1) / bs) * bs;
}

// 32 bytes to global memory in one store (sm_100 and later; 32-byte aligned
// address): a whole sector where a warp's store covers one row per thread.
__device__ __forceinline__ void st_global_v8(uint32_t* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Packed fp32 pairs (sm_100 and later: one instruction does the work of two,
// each half rounded as its scalar counterpart): (x, y) = (a0 b + c, a1 b + c)
// and (x, y) += (a0, a1).
__device__ __forceinline__ void ffma2(float& x, float& y, float a0, float a1, float b, float c) {
  asm("{\n.reg .b64 a, b, c, d;\nmov.b64 a, {%2, %3};\nmov.b64 b, {%4, %4};\n"
      "mov.b64 c, {%5, %5};\nfma.rn.f32x2 d, a, b, c;\nmov.b64 {%0, %1}, d;\n}"
      : "=f"(x), "=f"(y)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void fadd2(float& x, float& y, float a0, float a1) {
  asm("{\n.reg .b64 a, b;\nmov.b64 a, {%0, %1};\nmov.b64 b, {%2, %3};\n"
      "add.rn.f32x2 a, a, b;\nmov.b64 {%0, %1}, a;\n}"
      : "+f"(x), "+f"(y)
      : "f"(a0), "f"(a1));
}

// lo += the low bf16 half of pk, hi += its high half (each widened exactly,
// then one fp32 add): the row sums of the bf16-rounded softmax weights.
__device__ __forceinline__ void add_bf16x2_f32(float& lo, float& hi, uint32_t pk) {
  asm("{\n.reg .b16 l, h;\nmov.b32 {l, h}, %2;\nadd.rn.f32.bf16 %0, l, %0;\n"
      "add.rn.f32.bf16 %1, h, %1;\n}"
      : "+f"(lo), "+f"(hi)
      : "r"(pk));
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace pa
