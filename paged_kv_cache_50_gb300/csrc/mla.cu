// MLA latent decode ("Triton and MLA" (vllm-arch-zh), data-flow section):
// MQA over one latent KV head.  The cache row of a token is the 576-wide
// [kv_c (512) | k_pe (64)] vector; the key is the whole row, the value its
// first 512 entries, so every cache byte is read once for both products.
// Split-KV stage 1 here writes [B, H, S, 513] fp32 partials (LSE in the last
// slot); the LSE merge of decode.cu finishes the call.
//
// Warp-level tensor-core version (mma.m16n8k16):
//  * CTA = (group of 64 heads, split, request), 8 warps: warp w owns heads
//    16*(w % 4) .. +15 of the group and value columns 256*(w / 4) .. +255;
//  * Q of the 64 heads stays in shared memory (72 KB); 32-token cache tiles
//    (36 KB, contiguous within a 64-token block) stream through a
//    double-buffered cp.async ring;
//  * each warp computes S = Q K^T for its heads (the two column halves
//    recompute the same S), the online softmax, and O += P V for its 256
//    value columns.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

struct MlaCfg {
  static constexpr int kDk = 576;
  static constexpr int kDv = 512;
  static constexpr int kHeads = 64;               // heads per CTA
  static constexpr int kWarps = 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kBN = 32;                  // tokens per tile
  static constexpr int kRowBytes = kDk * 2;       // 1152
  static constexpr int kChunks = kDk / 8;         // 72
  static constexpr int kQBytes = kHeads * kRowBytes;
  static constexpr int kTileBytes = kBN * kRowBytes;
  static constexpr int kSmemBytes = kQBytes + 2 * kTileBytes;
};

__device__ __forceinline__ uint32_t mswz(int row, int chunk) {
  return static_cast<uint32_t>(row * MlaCfg::kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(256)
mla_decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ cache,
                  const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens,
                  int max_blocks, int H, int bs, int num_blocks, float scale_log2, int S,
                  int chunk, float* __restrict__ ws, int* err) {
  using C = MlaCfg;
  extern __shared__ __align__(128) uint8_t smem[];
  const int hg = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;
  const int hrow0 = (warp & 3) * 16;   // first head row of this warp within the CTA
  const int half = warp >> 2;          // value-column half

  const int seq = seq_lens[b];
  // Split s covers [s*chunk, (s+1)*chunk) (the last split runs to the end).
  const long long a0 = static_cast<long long>(s) * chunk;
  const int t0 = static_cast<int>(a0 < seq ? a0 : seq);
  const int t1 = (s == S - 1) ? seq : static_cast<int>(a0 + chunk < seq ? a0 + chunk : seq);
  const int ntiles = (t1 - t0 + C::kBN - 1) / C::kBN;

  const uint32_t qs = smem_u32(smem);
  const uint32_t kvs = qs + C::kQBytes;
  const int32_t* table = block_table + static_cast<int64_t>(b) * max_blocks;

  // Q of the 64 heads -> shared memory.
  {
    const __nv_bfloat16* qb = q + (static_cast<int64_t>(b) * H + hg * C::kHeads) * C::kDk;
    for (int c = threadIdx.x; c < C::kHeads * C::kChunks; c += C::kThreads) {
      const int r = c / C::kChunks, cc = c % C::kChunks;
      cp_async_16(qs + mswz(r, cc), qb + r * C::kDk + cc * 8, 16);
    }
  }
  auto issue = [&](int kt) {
    const uint32_t dst = kvs + (kt & 1) * C::kTileBytes;
    const int tb = t0 + kt * C::kBN;   // a multiple of 32, inside one block (bs % 64 == 0)
    const int blk = block_at(table, tb / bs, max_blocks);
    const bool ok = blk >= 0 && blk < num_blocks;
    if (!ok && threadIdx.x == 0) record_error(err, PA_DEVERR_BLOCK_ID);
    const __nv_bfloat16* src =
        cache + (static_cast<int64_t>(ok ? blk : 0) * bs + tb % bs) * C::kDk;
#pragma unroll
    for (int k = 0; k < C::kBN * C::kChunks / C::kThreads; ++k) {
      const int c = threadIdx.x + C::kThreads * k;
      const int r = c / C::kChunks, cc = c % C::kChunks;
      const int bytes = (ok && tb + r < t1) ? 16 : 0;
      cp_async_16(dst + mswz(r, cc), src + r * C::kDk + cc * 8, bytes);
    }
  };

  float m_r[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_r[2] = {0.f, 0.f};
  float o[32][4];
#pragma unroll
  for (int nd = 0; nd < 32; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;

  if (ntiles > 0) issue(0);
  cp_async_commit();
  for (int kt = 0; kt < ntiles; ++kt) {
    if (kt + 1 < ntiles) issue(kt + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const uint32_t kb = kvs + (kt & 1) * C::kTileBytes;
    const int tb = t0 + kt * C::kBN;
    const int blk = block_at(table, tb / bs, max_blocks);
    const int lim = (blk >= 0 && blk < num_blocks) ? min(C::kBN, t1 - tb) : 0;

    float sc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int qrow = hrow0 + (mi & 1) * 8 + rr;
#pragma unroll 4
      for (int kk = 0; kk < C::kDk / 16; ++kk) {
        uint32_t a[4];
        ldmatrix_x4(qs + mswz(qrow, 2 * kk + (mi >> 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int tok = np * 16 + (mi >> 1) * 8 + rr;
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kb + mswz(tok, 2 * kk + (mi & 1)), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * np], a, b0, b1);
          mma_bf16_16816(sc[2 * np + 1], a, b2, b3);
        }
      }
    }

    float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
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
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = fast_exp2(sc[nt][e] - mu[e >> 1]);
        sc[nt][e] = p;
        l_r[e >> 1] += p;
      }
#pragma unroll
    for (int nd = 0; nd < 32; ++nd) {
      o[nd][0] *= alpha[0];
      o[nd][1] *= alpha[0];
      o[nd][2] *= alpha[1];
      o[nd][3] *= alpha[1];
    }
    {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t pf[4];
        pf[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        pf[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        pf[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pf[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        const int tok = kk * 16 + (mi & 1) * 8 + rr;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(kb + mswz(tok, half * 32 + 2 * jj + (mi >> 1)), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * jj], pf, b0, b1);
          mma_bf16_16816(o[2 * jj + 1], pf, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = hg * C::kHeads + hrow0 + gid + 8 * r;
    float* dst = ws + ((static_cast<int64_t>(b) * H + h) * S + s) * (C::kDv + 1);
    const float inv = l_r[r] > 0.f ? 1.f / l_r[r] : 0.f;
#pragma unroll
    for (int nd = 0; nd < 32; ++nd) {
      const int col = half * 256 + nd * 8 + 2 * tid4;
      // Rows of the workspace are Dv + 1 = 513 floats: only 4-byte aligned.
      dst[col] = o[nd][2 * r] * inv;
      dst[col + 1] = o[nd][2 * r + 1] * inv;
    }
    if (half == 0 && tid4 == 0)
      dst[C::kDv] = l_r[r] > 0.f ? (m_r[r] + log2f(l_r[r])) * kLn2 : -CUDART_INF_F;
  }
}

cudaError_t launch_mla_decode(const void* q, const void* cache, const int32_t* block_table,
                              const int32_t* seq_lens, int B, int H, int bs, int num_blocks,
                              int max_blocks, float scale, int S, int chunk, float* ws, void* out,
                              float* lse, int* err, cudaStream_t stream) {
  using C = MlaCfg;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(mla_decode_kernel, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  dim3 grid(H / C::kHeads, S, B);
  mla_decode_kernel<<<grid, C::kThreads, C::kSmemBytes, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(cache), block_table,
      seq_lens, max_blocks, H, bs, num_blocks, scale * kLog2e, S, chunk, ws, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lse_merge(ws, B * H, S, C::kDv, out, lse, stream);
}

}  // namespace pa
