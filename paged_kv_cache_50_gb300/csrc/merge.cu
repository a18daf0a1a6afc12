// Split-KV decode, stage 2: the LSE merge of the split partials.
//
// Method: "Triton and MLA" (vllm-arch-zh), data flow -- each split leaves a
// partial output normalised within the split and its log-sum-exp in the
// workspace [N*H, S, dv + 1] (the "+1" slot); "Chapter 1: attention backends"
// (zero-to-sglang), section 3.1 -- the partials are combined with weights
// exp(lse_s - M), M = max_s lse_s:  o = sum_s w_s o_s / sum_s w_s and
// lse = M + ln sum_s w_s.  An empty split (lse = -inf) has weight 0; a row
// whose every split is empty gives o = 0 and lse = -inf.
//
// The partials were written by the kernel just before this one and sit in L2;
// the merge is latency-bound, not bandwidth-bound (8.5 MB for the 64-request
// GQA decode batch at 8 splits).  So for the common case of few splits
// (S <= 16 at dv = 128, S <= 32 at dv = 64) one warp serves one (request,
// head) and issues every load it needs -- the S LSEs (lane s holds split s)
// and the S x dv partial values (lane holds columns lane + 32 k) -- before any
// arithmetic: a single round trip to L2, then shuffles.  Every other shape
// takes the general kernel, one CTA per (request, head).
//
// Both kernels call pdl_trigger as soon as they start, so the next kernel of
// the stream (the following step's cache write) can be scheduled while the
// merge runs; every kernel launched with launch_pdl waits for its
// predecessor's completion before touching global memory.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

// Few splits: one warp per (request, head), four per CTA.  SMAX bounds S
// (registers: SMAX * DV / 32 floats per lane).
template <int DV, int SMAX>
__global__ void __launch_bounds__(128)
lse_merge_warp_kernel(const float* __restrict__ ws, int NH, int S, __nv_bfloat16* __restrict__ out,
                      float* __restrict__ lse) {
  static_assert(DV % 32 == 0 && SMAX <= 32, "lane layout");
  constexpr int kPer = DV / 32;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t nh = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (nh >= NH) return;   // whole warps only: nh is uniform within a warp
  const float* base = ws + nh * S * static_cast<int64_t>(DV + 1);

  const float l = lane < S ? base[static_cast<int64_t>(lane) * (DV + 1) + DV] : -CUDART_INF_F;
  float v[SMAX][kPer];
#pragma unroll
  for (int s = 0; s < SMAX; ++s)
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      v[s][k] = s < S ? base[static_cast<int64_t>(s) * (DV + 1) + k * 32 + lane] : 0.f;

  float m = l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float w = (m == -CUDART_INF_F || l == -CUDART_INF_F) ? 0.f : expf(l - m);
  float wsum = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const float inv = m == -CUDART_INF_F ? 0.f : 1.f / wsum;

  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
#pragma unroll
  for (int s = 0; s < SMAX; ++s) {
    if (s < S) {   // S is uniform, so the shuffle sees the whole warp
      const float ws_s = __shfl_sync(0xffffffffu, w, s);
#pragma unroll
      for (int k = 0; k < kPer; ++k) acc[k] += ws_s * v[s][k];
    }
  }
  __nv_bfloat16* dst = out + nh * DV;
#pragma unroll
  for (int k = 0; k < kPer; ++k) dst[k * 32 + lane] = __float2bfloat16_rn(acc[k] * inv);
  if (lse != nullptr && lane == 0) lse[nh] = m == -CUDART_INF_F ? -CUDART_INF_F : m + logf(wsum);
}

// Any number of splits and any width: one CTA per (request, head), the S
// weights exp(lse_s - M) kept in shared memory.
__global__ void __launch_bounds__(128)
lse_merge_kernel(const float* __restrict__ ws, int S, int dv, __nv_bfloat16* __restrict__ out,
                 float* __restrict__ lse) {
  extern __shared__ float wsh[];   // [S] weights, then 32 floats of reduction scratch
  float* red = wsh + S;
  pdl_wait();
  pdl_trigger();
  const int64_t nh = blockIdx.x;
  const float* base = ws + nh * S * static_cast<int64_t>(dv + 1);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  float m = -CUDART_INF_F;
  for (int s = tid; s < S; s += blockDim.x) m = fmaxf(m, base[static_cast<int64_t>(s) * (dv + 1) + dv]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  __syncthreads();

  float wsum = 0.f;
  for (int s = tid; s < S; s += blockDim.x) {
    const float l = base[static_cast<int64_t>(s) * (dv + 1) + dv];
    const float w = (m == -CUDART_INF_F || l == -CUDART_INF_F) ? 0.f : expf(l - m);
    wsh[s] = w;
    wsum += w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane == 0) red[8 + warp] = wsum;
  __syncthreads();
  wsum = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) wsum += red[8 + w];

  const float inv = m == -CUDART_INF_F ? 0.f : 1.f / wsum;
  for (int e = tid; e < dv; e += blockDim.x) {
    float acc = 0.f;
    int s = 0;
    for (; s + 4 <= S; s += 4) {
      const float* p = base + static_cast<int64_t>(s) * (dv + 1) + e;
      const float v0 = p[0], v1 = p[dv + 1], v2 = p[2 * (dv + 1)], v3 = p[3 * (dv + 1)];
      acc += wsh[s] * v0 + wsh[s + 1] * v1 + wsh[s + 2] * v2 + wsh[s + 3] * v3;
    }
    for (; s < S; ++s) acc += wsh[s] * base[static_cast<int64_t>(s) * (dv + 1) + e];
    out[nh * dv + e] = __float2bfloat16_rn(acc * inv);
  }
  if (lse != nullptr && tid == 0) lse[nh] = m == -CUDART_INF_F ? -CUDART_INF_F : m + logf(wsum);
}

template <int DV, int SMAX>
static cudaError_t launch_warp_merge(const float* ws, int NH, int S, void* out, float* lse,
                                     cudaStream_t stream) {
  return launch_pdl(lse_merge_warp_kernel<DV, SMAX>, dim3((NH + 3) / 4), dim3(128), 0, stream, ws,
                    NH, S, static_cast<__nv_bfloat16*>(out), lse);
}

cudaError_t launch_lse_merge(const float* ws, int NH, int S, int dv, void* out, float* lse,
                             cudaStream_t stream) {
  if (dv == 128 && S <= 8) return launch_warp_merge<128, 8>(ws, NH, S, out, lse, stream);
  if (dv == 128 && S <= 16) return launch_warp_merge<128, 16>(ws, NH, S, out, lse, stream);
  if (dv == 64 && S <= 16) return launch_warp_merge<64, 16>(ws, NH, S, out, lse, stream);
  if (dv == 64 && S <= 32) return launch_warp_merge<64, 32>(ws, NH, S, out, lse, stream);
  const size_t smem = (static_cast<size_t>(S) + 32) * sizeof(float);
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(lse_merge_kernel, 200 * 1024, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(lse_merge_kernel, dim3(NH), dim3(128), smem, stream, ws, S, dv,
                    static_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace pa
