// Split-KV decode (stage 1) and the LSE merge (stage 2) for the standard
// paged layout [num_blocks, 2, block_size, Hkv, d].
//
// Method: "Chapter 1: attention backends" (zero-to-sglang), section 3.1 --
// a decode query has too little parallelism, so the context is split along
// the sequence, each split yields a partial output with its softmax
// normaliser, and the partials are merged; section 4.1 -- inside a split the
// keys are consumed tile by tile with an online softmax (running max and sum,
// earlier output rescaled when the max grows, Fig. 5c).  Workspace layout
// [N, Hq, S, d + 1] with the LSE in the last slot: data-flow section of
// "Triton and MLA" (vllm-arch-zh).
//
// GB300 design (decode is HBM-bound: every K/V byte is read exactly once):
//  * one CTA per (split, kv head, request); its 4 warps take the split's
//    16-token sub-blocks round-robin, each warp with its own cp.async
//    pipeline (STAGES deep) into an XOR-swizzled shared-memory ring, so the
//    main loop has no CTA-wide barrier;
//  * all Hq/Hkv query heads of the kv group are the 16 rows of one
//    mma.m16n8k16 tile, so the K/V bytes fetched once serve the whole group:
//    S = Q K^T (16 x 16 per sub-block), online softmax in registers with quad
//    shuffles (exp2 with the scale folded in), O += P V;
//  * the four warps' (max, sum, O) states are merged through shared memory
//    at the end and the split's normalised partial and natural-log LSE are
//    written to the workspace.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

template <int D, int STAGES>
struct DecodeCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRowBytes = D * 2;            // one token of one head
  static constexpr int kChunks = D / 8;              // 16-byte chunks per row
  static constexpr int kTileBytes = 16 * kRowBytes;  // 16 tokens of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes; // K + V
  static constexpr int kWarpBytes = STAGES * kStageBytes;
  static constexpr int kPipeBytes = kWarps * kWarpBytes;
  static constexpr int kOStride = D + 4;             // padded fp32 row in the combine buffer
  static constexpr int kCombineBytes = kWarps * (16 * kOStride + 32) * 4;
  static constexpr int kSmemBytes = kPipeBytes > kCombineBytes ? kPipeBytes : kCombineBytes;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk, int row_bytes) {
  return static_cast<uint32_t>(row * row_bytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

template <int D, int STAGES>
__global__ void __launch_bounds__(128)
decode_splitkv_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ cache,
                      const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens,
                      int max_blocks, int Hq, int Hkv, int bs, int num_blocks, float scale_log2,
                      int S, int chunk, float* __restrict__ ws, int* err) {
  using C = DecodeCfg<D, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int s = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const int grp = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;

  // Every input may come from the previous kernel in the stream.
  pdl_wait();
  const int seq = seq_lens[i];
  // Split s covers [s*chunk, (s+1)*chunk) of the request (the last split runs
  // to the end), chunk being one block-aligned size for the whole batch.
  const long long a0 = static_cast<long long>(s) * chunk;
  const int t0 = static_cast<int>(a0 < seq ? a0 : seq);
  const int t1 = (s == S - 1) ? seq : static_cast<int>(a0 + chunk < seq ? a0 + chunk : seq);
  const int nsb = (t1 - t0 + 15) >> 4;
  const int my_n = nsb > warp ? (nsb - warp + C::kWarps - 1) / C::kWarps : 0;

  // Q of the kv group as the A operand: rows = the group's heads, zero-padded to 16.
  uint32_t qf[D / 16][4];
  {
    const __nv_bfloat16* qb = q + (static_cast<int64_t>(i) * Hq + static_cast<int64_t>(kvh) * grp) * D;
    const bool r0 = gid < grp, r1 = gid + 8 < grp;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c0 = kk * 16 + 2 * tid4;
      qf[kk][0] = r0 ? ld_u32(qb + gid * D + c0) : 0u;
      qf[kk][1] = r1 ? ld_u32(qb + (gid + 8) * D + c0) : 0u;
      qf[kk][2] = r0 ? ld_u32(qb + gid * D + c0 + 8) : 0u;
      qf[kk][3] = r1 ? ld_u32(qb + (gid + 8) * D + c0 + 8) : 0u;
    }
  }

  const uint32_t wbase = smem_u32(smem) + warp * C::kWarpBytes;
  const int64_t row_stride = static_cast<int64_t>(Hkv) * D;
  const int32_t* table = block_table + static_cast<int64_t>(i) * max_blocks;

  auto issue = [&](int n) {
    const int tb = t0 + (warp + n * C::kWarps) * 16;
    const int blk = block_at(table, tb / bs, max_blocks);
    const bool ok = blk >= 0 && blk < num_blocks;
    if (!ok && lane == 0) record_error(err, PA_DEVERR_BLOCK_ID);
    const int off = tb % bs;
    const __nv_bfloat16* kbase =
        cache + ((static_cast<int64_t>(ok ? blk : 0) * 2) * bs + off) * row_stride +
        static_cast<int64_t>(kvh) * D;
    const __nv_bfloat16* vbase = kbase + static_cast<int64_t>(bs) * row_stride;
    const uint32_t kdst = wbase + (n % STAGES) * C::kStageBytes;
    const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
    for (int k = 0; k < 16 * C::kChunks / 32; ++k) {
      const int c = lane + 32 * k;
      const int r = c / C::kChunks, cc = c % C::kChunks;
      const int bytes = (ok && tb + r < t1) ? 16 : 0;
      const uint32_t so = swz(r, cc, C::kRowBytes);
      cp_async_16(kdst + so, kbase + r * row_stride + cc * 8, bytes);
      cp_async_16(vdst + so, vbase + r * row_stride + cc * 8, bytes);
    }
  };

  float m_r[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_r[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;

#pragma unroll
  for (int n = 0; n < STAGES - 1; ++n) {
    if (n < my_n) issue(n);
    cp_async_commit();
  }

  for (int n = 0; n < my_n; ++n) {
    cp_async_wait<STAGES - 2>();
    __syncwarp();
    if (n + STAGES - 1 < my_n) issue(n + STAGES - 1);
    cp_async_commit();

    const int tb = t0 + (warp + n * C::kWarps) * 16;
    const int blk = block_at(table, tb / bs, max_blocks);
    const int lim = (blk >= 0 && blk < num_blocks) ? min(16, t1 - tb) : 0;
    const uint32_t kb = wbase + (n % STAGES) * C::kStageBytes;
    const uint32_t vb = kb + C::kTileBytes;

    // S = Q K^T: 16 heads x 16 tokens.
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int tok = (mi >> 1) * 8 + rr;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kb + swz(tok, 2 * kk + (mi & 1), C::kRowBytes), b0, b1, b2, b3);
        mma_bf16_16816(sc[0], qf[kk], b0, b1);
        mma_bf16_16816(sc[1], qf[kk], b2, b3);
      }
    }

    // Online softmax (log2 domain, scale folded in).
    float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = nt * 8 + 2 * tid4 + (e & 1);
        const float x = tok < lim ? sc[nt][e] * scale_log2 : -CUDART_INF_F;
        sc[nt][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    float alpha[2], mu[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m_r[r], mx[r]);
      mu[r] = mn == -CUDART_INF_F ? 0.f : mn;
      alpha[r] = fast_exp2(m_r[r] - mu[r]);
      m_r[r] = mn;
      l_r[r] *= alpha[r];
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = fast_exp2(sc[nt][e] - mu[e >> 1]);
        sc[nt][e] = p;
        l_r[e >> 1] += p;
      }
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o[nd][0] *= alpha[0];
      o[nd][1] *= alpha[0];
      o[nd][2] *= alpha[1];
      o[nd][3] *= alpha[1];
    }
    uint32_t pf[4];
    pf[0] = pack_bf16(sc[0][0], sc[0][1]);
    pf[1] = pack_bf16(sc[0][2], sc[0][3]);
    pf[2] = pack_bf16(sc[1][0], sc[1][1]);
    pf[3] = pack_bf16(sc[1][2], sc[1][3]);

    // O += P V.
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int tok = (mi & 1) * 8 + rr;
#pragma unroll
      for (int jj = 0; jj < D / 16; ++jj) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vb + swz(tok, 2 * jj + (mi >> 1), C::kRowBytes), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * jj], pf, b0, b1);
        mma_bf16_16816(o[2 * jj + 1], pf, b2, b3);
      }
    }
  }
  cp_async_wait<0>();
  // The merge may start launching (it waits for this kernel to complete).
  pdl_trigger();

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
  }

  // Merge the four warps' states through shared memory.
  __syncthreads();
  float* cbuf = reinterpret_cast<float*>(smem);
  float* mbuf = cbuf + C::kWarps * 16 * C::kOStride;  // [warp][16]
  float* lbuf = mbuf + C::kWarps * 16;                // [warp][16]
  {
    float* ob = cbuf + warp * 16 * C::kOStride;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const int col = nd * 8 + 2 * tid4;
      *reinterpret_cast<float2*>(ob + gid * C::kOStride + col) = make_float2(o[nd][0], o[nd][1]);
      *reinterpret_cast<float2*>(ob + (gid + 8) * C::kOStride + col) =
          make_float2(o[nd][2], o[nd][3]);
    }
    if (tid4 == 0) {
      mbuf[warp * 16 + gid] = m_r[0];
      mbuf[warp * 16 + gid + 8] = m_r[1];
      lbuf[warp * 16 + gid] = l_r[0];
      lbuf[warp * 16 + gid + 8] = l_r[1];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < grp * D; idx += C::kThreads) {
    const int r = idx / D, e = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mbuf[w * 16 + r]);
    float* dst = ws + ((static_cast<int64_t>(i) * Hq + kvh * grp + r) * S + s) * (D + 1);
    if (M == -CUDART_INF_F) {
      dst[e] = 0.f;
      if (e == 0) dst[D] = -CUDART_INF_F;
      continue;
    }
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) {
      const float f = fast_exp2(mbuf[w * 16 + r] - M);
      L += f * lbuf[w * 16 + r];
      acc += f * cbuf[(w * 16 + r) * C::kOStride + e];
    }
    dst[e] = acc / L;
    if (e == 0) dst[D] = (M + log2f(L)) * kLn2;
  }
}

// Stage 2: one CTA per (request, head); weights exp(lse_s - M) in shared memory.
__global__ void __launch_bounds__(128)
lse_merge_kernel(const float* __restrict__ ws, int S, int dv, __nv_bfloat16* __restrict__ out,
                 float* __restrict__ lse) {
  extern __shared__ float wsh[];   // [S] weights, then 32 floats of reduction scratch
  float* red = wsh + S;
  pdl_wait();
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

template <int D, int STAGES>
static cudaError_t launch_decode_t(const void* q, const void* cache, const int32_t* block_table,
                                   const int32_t* seq_lens, int N, int Hq, int Hkv, int bs,
                                   int num_blocks, int max_blocks, float scale, int S, int chunk,
                                   float* ws, int* err, cudaStream_t stream) {
  using C = DecodeCfg<D, STAGES>;
  auto kern = decode_splitkv_kernel<D, STAGES>;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(kern, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(S, Hkv, N), dim3(C::kThreads), C::kSmemBytes, stream,
                    static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(cache),
                    block_table, seq_lens, max_blocks, Hq, Hkv, bs, num_blocks, scale * kLog2e, S,
                    chunk, ws, err);
}

cudaError_t launch_decode_splitkv(const void* q, const void* cache, const int32_t* block_table,
                                  const int32_t* seq_lens, int N, int Hq, int Hkv, int d, int bs,
                                  int num_blocks, int max_blocks, float scale, int S, int chunk,
                                  float* ws, int* err, cudaStream_t stream) {
  if (d == 128)
    return launch_decode_t<128, 2>(q, cache, block_table, seq_lens, N, Hq, Hkv, bs, num_blocks,
                                   max_blocks, scale, S, chunk, ws, err, stream);
  return launch_decode_t<64, 4>(q, cache, block_table, seq_lens, N, Hq, Hkv, bs, num_blocks,
                                max_blocks, scale, S, chunk, ws, err, stream);
}

cudaError_t launch_lse_merge(const float* ws, int NH, int S, int dv, void* out, float* lse,
                             cudaStream_t stream) {
  const size_t smem = (static_cast<size_t>(S) + 32) * sizeof(float);
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(lse_merge_kernel, 200 * 1024, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(lse_merge_kernel, dim3(NH), dim3(128), smem, stream, ws, S, dv,
                    static_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace pa
